"""Python binding of libmfr.so — MoE finalize + residual + RMSNorm on GB300.

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI (include/moe_finalize_rmsnorm.h).  PyTorch supplies
device memory and streams.  There is no CPU fallback: if the library is not
built, importing the binding's entry points raises.

    import moe_finalize_residual_rmsnorm_gb300 as mfr
    plan = mfr.Plan(T, H, k, R)
    plan.run(expert_out, permuted_row_of, topk_weights, residual_in,
             residual_out, gamma, eps, out)          # current torch stream
"""
from __future__ import annotations

import collections
import ctypes
import os
from typing import Optional

from .build import LIBRARY, build as _build_library

__all__ = [
    "LIBRARY", "MFRError", "Plan", "FinalizePlan", "Nvfp4Plan", "ExpertNormPlan", "PlanInfo", "Options", "build", "load_library", "supports",
    "moe_finalize_residual_rmsnorm", "finalize_residual_rmsnorm_host", "exported_symbols",
    "run_noalloc", "validate_fused_args", "SF_ROW_MAJOR", "SF_TILED_128x4", "VARIANT_AUTO", "VARIANT_CLUSTER", "VARIANT_ROWS", "VARIANT_STREAM", "STATUS_BAD_INDEX",
    "ERROR_CODES",
]

MFR_OK = 0
ERROR_CODES = {
    1: "MFR_ERR_INVALID_ARG", 2: "MFR_ERR_UNSUPPORTED_SHAPE", 3: "MFR_ERR_MISALIGNED",
    4: "MFR_ERR_BAD_DEVICE", 5: "MFR_ERR_LAUNCH", 6: "MFR_ERR_CUDA", 7: "MFR_ERR_BAD_INDEX",
}
STATUS_BAD_INDEX = 1
STATUS_TIMEOUT = 2
SF_ROW_MAJOR, SF_TILED_128x4 = 0, 1
FLOOR_LOAD, FLOOR_EXCHANGE, FLOOR_STORE = 1, 2, 4
VARIANT_AUTO, VARIANT_CLUSTER, VARIANT_ROWS, VARIANT_STREAM = 0, 1, 2, 3
VARIANT_NAMES = {VARIANT_CLUSTER: "cluster", VARIANT_ROWS: "rows", VARIANT_STREAM: "stream"}


class MFRError(RuntimeError):
    def __init__(self, code: int, where: str, detail: str):
        self.code = code
        self.name = ERROR_CODES.get(code, f"code {code}")
        super().__init__(f"{where}: {self.name}: {detail}")


class Options(ctypes.Structure):
    _fields_ = [("enable_pdl", ctypes.c_int), ("force_variant", ctypes.c_int),
                ("cluster_size", ctypes.c_int), ("debug_checks", ctypes.c_int),
                ("sentinel_skip", ctypes.c_int)]


class PlanInfo(ctypes.Structure):
    _fields_ = [("variant", ctypes.c_int), ("grid_x", ctypes.c_int), ("grid_y", ctypes.c_int),
                ("block", ctypes.c_int), ("cluster", ctypes.c_int), ("smem_bytes", ctypes.c_int),
                ("chunks_per_thread", ctypes.c_int), ("sm_count", ctypes.c_int), ("slot_registers", ctypes.c_int)]

    def as_dict(self):
        d = {name: getattr(self, name) for name, _ in self._fields_}
        d["variant_name"] = VARIANT_NAMES.get(self.variant, "?")
        return d


# (name, restype, argtypes) of every symbol the header declares
_VP, _I64, _I, _F = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
SIGNATURES = {
    "moe_finalize_rmsnorm_supports": (_I, [_I64, _I]),
    "moe_finalize_rmsnorm_default_options": (None, [ctypes.POINTER(Options)]),
    "moe_finalize_rmsnorm_plan": (_I, [ctypes.POINTER(_VP), _I64, _I64, _I, _I64, ctypes.POINTER(Options)]),
    "moe_finalize_rmsnorm_run": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _F, _VP, _VP]),
    "moe_finalize_rmsnorm_get_status": (_I, [_VP, _VP, ctypes.POINTER(_I)]),
    "moe_finalize_rmsnorm_plan_info": (_I, [_VP, ctypes.POINTER(PlanInfo)]),
    "moe_finalize_rmsnorm_launch_floor": (_I, [_VP, _VP]),
    "moe_finalize_rmsnorm_launch_floor_work": (_I, [_VP, _I, _VP, _VP, _VP, _VP, _VP, _VP]),
    "moe_finalize_rmsnorm_wait_selftest": (_I, [_VP, ctypes.c_int64, ctypes.c_int, _VP]),
    "moe_finalize_rmsnorm_bench_producer": (_I, [_VP, _VP, _I64, _I64, ctypes.c_longlong, _I, _VP]),
    "moe_finalize_rmsnorm_host_workspace_bytes": (_I64, [_VP]),
    "moe_finalize_rmsnorm_run_host": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _F, _VP, _VP, _I64, _VP]),
    "moe_finalize_rmsnorm_nvfp4_plan": (_I, [ctypes.POINTER(_VP), _I64, _I64, _I, _I64, ctypes.POINTER(Options)]),
    "moe_finalize_rmsnorm_nvfp4_run": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _F, _F, _VP, _VP, _VP]),
    "moe_finalize_rmsnorm_nvfp4_plan_ex": (_I, [ctypes.POINTER(_VP), _I64, _I64, _I, _I64, ctypes.POINTER(Options),
                                                 _I]),
    "moe_finalize_rmsnorm_nvfp4_sf_bytes": (_I64, [_VP]),
    "moe_finalize_plan": (_I, [ctypes.POINTER(_VP), _I64, _I64, _I, _I64, ctypes.POINTER(Options)]),
    "moe_finalize_run": (_I, [_VP, _VP, _VP, _VP, _VP, _VP]),
    "moe_finalize_expert_rmsnorm_plan": (_I, [ctypes.POINTER(_VP), _I64, _I64, _I, _I64, ctypes.POINTER(Options)]),
    "moe_finalize_expert_rmsnorm_run": (_I, [_VP, _VP, _VP, _VP, _VP, _F, _VP, _VP]),
    "moe_finalize_rmsnorm_run_noalloc": (_I, [_I64, _I64, _I, _I64, _VP, _VP, _VP, _VP, _VP, _VP, _F, _VP, _I,
                                               ctypes.POINTER(_I), _VP]),
    "moe_finalize_rmsnorm_destroy": (None, [_VP]),
    "moe_finalize_rmsnorm_strerror": (ctypes.c_char_p, [_I]),
    "moe_finalize_rmsnorm_last_error": (ctypes.c_char_p, []),
}

_lib = None


def build(force: bool = False, verbose: bool = False) -> str:
    """Compiles libmfr.so for sm_103a (nvcc) into the package directory."""
    return _build_library(force=force, verbose=verbose)


def load_library():
    """Loads the in-tree libmfr.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIBRARY):
            raise ImportError(f"{LIBRARY} is missing: build it with "
                              "moe_finalize_residual_rmsnorm_gb300.build() (nvcc, sm_103a)")
        lib = ctypes.CDLL(LIBRARY)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def exported_symbols():
    lib = load_library()
    return {name for name in SIGNATURES if hasattr(lib, name)}


def _check(code: int, where: str):
    if code != MFR_OK:
        lib = load_library()
        detail = lib.moe_finalize_rmsnorm_last_error().decode() or \
            lib.moe_finalize_rmsnorm_strerror(code).decode()
        raise MFRError(code, where, detail)


def supports(H: int, k: int) -> bool:
    return bool(load_library().moe_finalize_rmsnorm_supports(H, k))


def validate_fused_args(T: int, H: int, k: int, R: int, expert_out, permuted_row_of, topk_weights, residual_in,
                        residual_out, gamma, out) -> None:
    """Checks the tensors of one fused call against (T, H, k, R): dtype and
    shape of every tensor first, then contiguity, then that each is a CUDA
    tensor.  Raises ValueError on the first mismatch.  The C ABI receives
    bare pointers and cannot check sizes, so this is what keeps a wrongly
    sized or strided tensor from being read or written out of bounds."""
    import torch
    want = [
        ("expert_out", expert_out, torch.bfloat16, (R, H)),
        ("permuted_row_of", permuted_row_of, torch.int32, (T, k)),
        ("topk_weights", topk_weights, torch.float32, (T, k)),
        ("residual_in", residual_in, torch.float32, (T, H)),
        ("residual_out", residual_out, torch.float32, (T, H)),
        ("gamma", gamma, torch.bfloat16, (H,)),
        ("out", out, torch.bfloat16, (T, H)),
    ]
    for name, t, dt, shape in want:
        if not isinstance(t, torch.Tensor):
            raise ValueError(f"{name} must be a torch.Tensor, got {type(t).__name__}")
        if t.dtype != dt or tuple(t.shape) != shape:
            raise ValueError(f"{name}: expected {dt} {shape}, got {t.dtype} {tuple(t.shape)}")
    for name, t, _, _ in want:
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    for name, t, _, _ in want:
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    return t.data_ptr()


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class Plan:
    """A plan for T tokens, hidden size H, top-k k and R rows of expert_out on
    the current CUDA device (C: moe_finalize_rmsnorm_plan)."""

    _PLAN_FN = "moe_finalize_rmsnorm_plan"

    def __init__(self, T: int, H: int, k: int, R: Optional[int] = None, *, enable_pdl: bool = True,
                 variant: int = VARIANT_AUTO, cluster_size: int = 0, debug_checks: bool = False,
                 sentinel_skip: bool = False):
        lib = load_library()
        self._lib = lib
        self.T, self.H, self.k = int(T), int(H), int(k)
        self.R = int(T) * int(k) if R is None else int(R)
        opt = Options(int(bool(enable_pdl)), int(variant), int(cluster_size), int(bool(debug_checks)),
                      int(bool(sentinel_skip)))
        h = ctypes.c_void_p()
        _check(getattr(lib, self._PLAN_FN)(ctypes.byref(h), self.T, self.H, self.k, self.R,
                                           ctypes.byref(opt)), self._PLAN_FN)
        self._h = h

    @property
    def handle(self):
        return self._h

    def info(self) -> dict:
        inf = PlanInfo()
        _check(self._lib.moe_finalize_rmsnorm_plan_info(self._h, ctypes.byref(inf)), "plan_info")
        return inf.as_dict()

    def _validate(self, expert_out, permuted_row_of, topk_weights, residual_in, residual_out, gamma, out):
        validate_fused_args(self.T, self.H, self.k, self.R, expert_out, permuted_row_of, topk_weights, residual_in,
                            residual_out, gamma, out)

    def run(self, expert_out, permuted_row_of, topk_weights, residual_in, residual_out, gamma,
            eps: float, out, stream=None, *, validate: bool = True) -> None:
        """Enqueues one call on `stream` (default: torch's current stream).
        residual_out may be residual_in (in place)."""
        if validate:
            self._validate(expert_out, permuted_row_of, topk_weights, residual_in, residual_out, gamma, out)
        code = self._lib.moe_finalize_rmsnorm_run(
            self._h, _ptr(expert_out), _ptr(permuted_row_of), _ptr(topk_weights), _ptr(residual_in),
            _ptr(residual_out), _ptr(gamma), ctypes.c_float(eps), _ptr(out), _stream_handle(stream))
        _check(code, "moe_finalize_rmsnorm_run")

    def run_ptrs(self, expert_out, permuted_row_of, topk_weights, residual_in, residual_out, gamma,
                 eps, out, stream) -> int:
        """Raw-pointer call (ints); returns the C return code unchanged."""
        return self._lib.moe_finalize_rmsnorm_run(self._h, expert_out, permuted_row_of, topk_weights,
                                                  residual_in, residual_out, gamma, ctypes.c_float(eps),
                                                  out, stream)

    def wait_selftest(self, limit_cycles: int, arrive: bool, stream=None) -> None:
        """One bounded on-chip wait that runs out unless `arrive`; a wait that
        runs out sets STATUS_TIMEOUT in the plan's status word
        (C: moe_finalize_rmsnorm_wait_selftest)."""
        _check(self._lib.moe_finalize_rmsnorm_wait_selftest(self._h, int(limit_cycles), int(bool(arrive)),
                                                            _stream_handle(stream)),
               "moe_finalize_rmsnorm_wait_selftest")

    def launch_floor(self, stream=None) -> None:
        """Enqueues the empty kernel with this plan's launch geometry."""
        _check(self._lib.moe_finalize_rmsnorm_launch_floor(self._h, _stream_handle(stream)),
               "moe_finalize_rmsnorm_launch_floor")

    def launch_floor_work(self, work: int, expert_out=None, permuted_row_of=None, residual_in=None,
                          residual_out=None, out=None, stream=None) -> None:
        """Enqueues the empty kernel with this plan's launch geometry plus the
        call's loads, a cluster barrier and/or its stores (FLOOR_* bits;
        C: moe_finalize_rmsnorm_launch_floor_work)."""
        _check(self._lib.moe_finalize_rmsnorm_launch_floor_work(
            self._h, int(work), _ptr(expert_out), _ptr(permuted_row_of), _ptr(residual_in), _ptr(residual_out),
            _ptr(out), _stream_handle(stream)), "moe_finalize_rmsnorm_launch_floor_work")

    def host_workspace_bytes(self) -> int:
        return int(self._lib.moe_finalize_rmsnorm_host_workspace_bytes(self._h))

    def run_host(self, expert_out, permuted_row_of, topk_weights, residual_in, residual_out, gamma, eps: float,
                 out, workspace, stream=None) -> None:
        """End to end from host tensors (pinned for asynchronous copies):
        inputs copied into `workspace` (a device uint8 tensor of at least
        host_workspace_bytes()), the kernel, outputs copied back, all on
        `stream` (C: moe_finalize_rmsnorm_run_host)."""
        for name, t in (("expert_out", expert_out), ("permuted_row_of", permuted_row_of),
                        ("topk_weights", topk_weights), ("residual_in", residual_in),
                        ("residual_out", residual_out), ("gamma", gamma), ("out", out)):
            if t.is_cuda or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous host tensor")
        code = self._lib.moe_finalize_rmsnorm_run_host(
            self._h, _ptr(expert_out), _ptr(permuted_row_of), _ptr(topk_weights), _ptr(residual_in),
            _ptr(residual_out), _ptr(gamma), ctypes.c_float(eps), _ptr(out), _ptr(workspace),
            workspace.numel() * workspace.element_size(), _stream_handle(stream))
        _check(code, "moe_finalize_rmsnorm_run_host")

    def get_status(self, stream=None) -> int:
        st = ctypes.c_int(0)
        _check(self._lib.moe_finalize_rmsnorm_get_status(self._h, _stream_handle(stream), ctypes.byref(st)),
               "moe_finalize_rmsnorm_get_status")
        return st.value

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            self._lib.moe_finalize_rmsnorm_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()


class Nvfp4Plan(Plan):
    """Residual + RMSNorm with the normalised output written as NVFP4
    (C: moe_finalize_rmsnorm_nvfp4_plan_ex / moe_finalize_rmsnorm_nvfp4_run):
    out_q uint8 [T, H/2] (two E2M1 codes per byte, even column in the low
    nibble), out_sf the E4M3 block scales, uint8 [T, H/16] row-major
    (sf_layout=SF_ROW_MAJOR) or sf_bytes() bytes in the 128 x 4 tiles that
    block-scaled FP4 GEMMs read (SF_TILED_128x4); s_enc the FP32 tensor
    scale."""

    _PLAN_FN = "moe_finalize_rmsnorm_nvfp4_plan"

    def __init__(self, T: int, H: int, k: int, R: Optional[int] = None, *, sf_layout: int = SF_ROW_MAJOR,
                 enable_pdl: bool = True, variant: int = VARIANT_AUTO, cluster_size: int = 0,
                 debug_checks: bool = False, sentinel_skip: bool = False):
        lib = load_library()
        self._lib = lib
        self.T, self.H, self.k = int(T), int(H), int(k)
        self.R = int(T) * int(k) if R is None else int(R)
        self.sf_layout = int(sf_layout)
        opt = Options(int(bool(enable_pdl)), int(variant), int(cluster_size), int(bool(debug_checks)),
                      int(bool(sentinel_skip)))
        h = ctypes.c_void_p()
        _check(lib.moe_finalize_rmsnorm_nvfp4_plan_ex(ctypes.byref(h), self.T, self.H, self.k, self.R,
                                                      ctypes.byref(opt), self.sf_layout),
               "moe_finalize_rmsnorm_nvfp4_plan_ex")
        self._h = h

    def sf_bytes(self) -> int:
        """Bytes of out_sf in this plan's layout."""
        return int(self._lib.moe_finalize_rmsnorm_nvfp4_sf_bytes(self._h))

    def run(self, expert_out, permuted_row_of, topk_weights, residual_in, residual_out, gamma, eps: float,
            s_enc: float, out_q, out_sf, stream=None, *, validate: bool = True):
        if validate:
            import torch
            T, H, k, R = self.T, self.H, self.k, self.R
            for name, t, dt, shape in [("expert_out", expert_out, torch.bfloat16, (R, H)),
                                       ("permuted_row_of", permuted_row_of, torch.int32, (T, k)),
                                       ("topk_weights", topk_weights, torch.float32, (T, k)),
                                       ("residual_in", residual_in, torch.float32, (T, H)),
                                       ("residual_out", residual_out, torch.float32, (T, H)),
                                       ("gamma", gamma, torch.bfloat16, (H,)),
                                       ("out_q", out_q, torch.uint8, (T, H // 2))] + \
                    ([("out_sf", out_sf, torch.uint8, (T, H // 16))] if self.sf_layout == SF_ROW_MAJOR else []):
                if t.dtype != dt or tuple(t.shape) != shape or not t.is_cuda or not t.is_contiguous():
                    raise ValueError(f"{name}: expected contiguous CUDA {dt} {shape}")
            if self.sf_layout != SF_ROW_MAJOR and (out_sf.dtype != torch.uint8 or out_sf.numel() != self.sf_bytes()
                                                   or not out_sf.is_cuda or not out_sf.is_contiguous()):
                raise ValueError(f"out_sf: expected a contiguous CUDA uint8 tensor of {self.sf_bytes()} bytes "
                                 "(the tiled block-scale layout)")
        code = self._lib.moe_finalize_rmsnorm_nvfp4_run(
            self._h, _ptr(expert_out), _ptr(permuted_row_of), _ptr(topk_weights), _ptr(residual_in),
            _ptr(residual_out), _ptr(gamma), ctypes.c_float(eps), ctypes.c_float(s_enc), _ptr(out_q),
            _ptr(out_sf), _stream_handle(stream))
        _check(code, "moe_finalize_rmsnorm_nvfp4_run")


class FinalizePlan(Plan):
    """Plain finalize, out = bf16(FP32 weighted sum), no residual and no norm
    (C: moe_finalize_plan / moe_finalize_run)."""

    _PLAN_FN = "moe_finalize_plan"

    def run(self, expert_out, permuted_row_of, topk_weights, out, stream=None, *, validate: bool = True):
        if validate:
            import torch
            for name, t, dt, shape in [("expert_out", expert_out, torch.bfloat16, (self.R, self.H)),
                                       ("permuted_row_of", permuted_row_of, torch.int32, (self.T, self.k)),
                                       ("topk_weights", topk_weights, torch.float32, (self.T, self.k)),
                                       ("out", out, torch.bfloat16, (self.T, self.H))]:
                if t.dtype != dt or tuple(t.shape) != shape or not t.is_cuda or not t.is_contiguous():
                    raise ValueError(f"{name}: expected contiguous CUDA {dt} {shape}")
        code = self._lib.moe_finalize_run(self._h, _ptr(expert_out), _ptr(permuted_row_of), _ptr(topk_weights),
                                          _ptr(out), _stream_handle(stream))
        _check(code, "moe_finalize_run")


class ExpertNormPlan(Plan):
    """Finalize with an RMSNorm per expert row before the weighted sum:
    out = bf16(sum_j w_j * ((E[r_j] * rsqrt(mean(E[r_j]^2) + eps)) * gamma)),
    no residual (C: moe_finalize_expert_rmsnorm_plan / _run)."""

    _PLAN_FN = "moe_finalize_expert_rmsnorm_plan"

    def run(self, expert_out, permuted_row_of, topk_weights, gamma, eps: float, out, stream=None, *,
            validate: bool = True):
        if validate:
            import torch
            for name, t, dt, shape in [("expert_out", expert_out, torch.bfloat16, (self.R, self.H)),
                                       ("permuted_row_of", permuted_row_of, torch.int32, (self.T, self.k)),
                                       ("topk_weights", topk_weights, torch.float32, (self.T, self.k)),
                                       ("gamma", gamma, torch.bfloat16, (self.H,)),
                                       ("out", out, torch.bfloat16, (self.T, self.H))]:
                if t.dtype != dt or tuple(t.shape) != shape or not t.is_cuda or not t.is_contiguous():
                    raise ValueError(f"{name}: expected contiguous CUDA {dt} {shape}")
        code = self._lib.moe_finalize_expert_rmsnorm_run(self._h, _ptr(expert_out), _ptr(permuted_row_of),
                                                         _ptr(topk_weights), _ptr(gamma), ctypes.c_float(eps),
                                                         _ptr(out), _stream_handle(stream))
        _check(code, "moe_finalize_expert_rmsnorm_run")


def bench_producer(src, expert_out, busy_cycles: int = 0, enable_pdl: bool = True, stream=None) -> None:
    """Stand-in for the GEMM2 producer (C: moe_finalize_rmsnorm_bench_producer):
    wait, signal dependents, stay busy, then copy src into expert_out."""
    lib = load_library()
    R, H = expert_out.shape
    _check(lib.moe_finalize_rmsnorm_bench_producer(_ptr(src), _ptr(expert_out), R, H, int(busy_cycles),
                                                   int(bool(enable_pdl)), _stream_handle(stream)),
           "moe_finalize_rmsnorm_bench_producer")


NOALLOC_SLOTS = 64


def run_noalloc(expert_out, permuted_row_of, topk_weights, residual_in, residual_out, gamma, eps: float, out,
                *, slot: int = 0, report_status: bool = False, stream=None, validate: bool = True):
    """Allocation-free call (C: moe_finalize_rmsnorm_run_noalloc): no plan, no
    device allocation; the status word is slot `slot` of the library's static
    scratch.  T, H, k and R are taken from permuted_row_of [T, k] and
    expert_out [R, H], and every other tensor is checked against them
    (validate_fused_args) before the C call.  Returns the status bits when
    report_status (the call then waits for the stream), else None."""
    if validate:
        if permuted_row_of.dim() != 2 or expert_out.dim() != 2:
            raise ValueError("permuted_row_of must be [T, k] and expert_out [R, H]")
        T, k = permuted_row_of.shape
        R, H = expert_out.shape
        validate_fused_args(T, H, k, R, expert_out, permuted_row_of, topk_weights, residual_in, residual_out,
                            gamma, out)
    lib = load_library()
    T, k = permuted_row_of.shape
    R, H = expert_out.shape
    st = ctypes.c_int(0)
    code = lib.moe_finalize_rmsnorm_run_noalloc(
        T, H, k, R, _ptr(expert_out), _ptr(permuted_row_of), _ptr(topk_weights), _ptr(residual_in),
        _ptr(residual_out), _ptr(gamma), ctypes.c_float(eps), _ptr(out), int(slot),
        ctypes.byref(st) if report_status else None, _stream_handle(stream))
    _check(code, "moe_finalize_rmsnorm_run_noalloc")
    return st.value if report_status else None


PLAN_CACHE_SIZE = 64
_plan_cache: "collections.OrderedDict" = collections.OrderedDict()


def cached_plan(T: int, H: int, k: int, R: int, **plan_kw) -> Plan:
    """The plan for (current device, T, H, k, R, options), made once and kept
    in a per-process cache of the PLAN_CACHE_SIZE most recently used plans.
    Plans are immutable, so one may serve calls on several streams.  A plan
    holds one device status word: an evicted plan is destroyed after its
    device has finished all queued work.  Make the plan before a CUDA graph
    capture, and keep plans that a graph uses outside the cache (Plan(...)),
    since a graph must not outlive its plans."""
    import torch
    key = (torch.cuda.current_device(), int(T), int(H), int(k), int(R), tuple(sorted(plan_kw.items())))
    plan = _plan_cache.get(key)
    if plan is None:
        plan = Plan(T, H, k, R, **plan_kw)
        _plan_cache[key] = plan
        while len(_plan_cache) > PLAN_CACHE_SIZE:
            (dev, *_), old = _plan_cache.popitem(last=False)
            torch.cuda.synchronize(dev)     # no run of the old plan is still in flight
            old.close()
    else:
        _plan_cache.move_to_end(key)
    return plan


def moe_finalize_residual_rmsnorm(expert_out, permuted_row_of, topk_weights, residual, gamma, eps: float,
                                  *, residual_out=None, out=None, stream=None, plan: Optional[Plan] = None,
                                  **plan_kw):
    """Allocating convenience wrapper: returns (residual_out, out).  With
    residual_out=residual the update is in place.  Without `plan` it takes
    the cached plan for the shapes and options (cached_plan)."""
    import torch
    T, k = permuted_row_of.shape
    R, H = expert_out.shape
    if residual_out is None:
        residual_out = torch.empty_like(residual)
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=residual.device)
    if plan is None:
        plan = cached_plan(T, H, k, R, **plan_kw)
    plan.run(expert_out, permuted_row_of, topk_weights, residual, residual_out, gamma, eps, out, stream)
    return residual_out, out


def finalize_residual_rmsnorm_host(plan: Plan, host_in: dict, host_out: dict, workspace, stream=None):
    """One end-to-end call on host buffers through the C ABI
    (moe_finalize_rmsnorm_run_host).  Returns (h2d_bytes, d2h_bytes) moved."""
    plan.run_host(host_in["expert_out"], host_in["permuted_row_of"], host_in["topk_weights"], host_in["residual"],
                  host_out["residual_out"], host_in["gamma"], host_in["eps"], host_out["out"], workspace, stream)
    h2d = sum(host_in[k].numel() * host_in[k].element_size()
              for k in ("expert_out", "permuted_row_of", "topk_weights", "residual", "gamma"))
    d2h = sum(host_out[k].numel() * host_out[k].element_size() for k in ("residual_out", "out"))
    return h2d, d2h
