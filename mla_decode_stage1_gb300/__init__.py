"""Python binding of libmla_decode (single-token MLA decode for GB300, sm_103a).

Argument marshalling only: every step of the decode runs in the library's
CUDA kernels.  The names mirror the C ABI in include/mla_decode.h:
``mla_decode_plan``, ``mla_decode_run``, ``mla_decode_check``,
``mla_status_string``.  PyTorch tensors are accepted for device memory and
``torch.cuda`` streams; there is no CPU fallback -- importing this package
fails loudly when the shared library has not been built.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmla_decode.so")

HEADS, QK_DIM, V_DIM, TILE = 16, 576, 512, 128
DTYPES = {"bf16": 0, "fp8": 1, "mxfp4": 2}
STATUS = {0: "MLA_OK", 1: "MLA_ERR_INVALID_ARG", 2: "MLA_ERR_UNSUPPORTED", 3: "MLA_ERR_WORKSPACE",
          4: "MLA_ERR_CUDA", 5: "MLA_ERR_DEVICE_TIMEOUT"}
EXPORTS = ("mla_decode_plan", "mla_decode_plan_q", "mla_decode_plan_ex", "mla_plan_workspace_size",
           "mla_plan_get_info", "mla_plan_get_work", "mla_plan_destroy", "mla_decode_run",
           "mla_decode_check", "mla_status_string", "mla_plan_set_stage1_events",
           "mla_decode_run_noalloc", "mla_selftest_bounded_wait", "mla_decode_autotune",
           "mla_autotune_select")


class MlaError(RuntimeError):
    def __init__(self, call: str, status: int):
        super().__init__(f"{call} failed: {STATUS.get(status, status)}")
        self.status = status


class PlanInfo(ctypes.Structure):
    _fields_ = [("batch_size", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("num_ctas", ctypes.c_int32), ("num_items", ctypes.c_int32),
                ("num_partials", ctypes.c_int32), ("num_merge_jobs", ctypes.c_int32),
                ("total_tokens", ctypes.c_int64), ("total_tiles", ctypes.c_int64),
                ("workspace_bytes", ctypes.c_size_t), ("q_len", ctypes.c_int32),
                ("unit_tokens", ctypes.c_int32), ("item_cost", ctypes.c_int32),
                ("cluster_size", ctypes.c_int32)]


class PlanOptions(ctypes.Structure):
    _fields_ = [("num_splits", ctypes.c_int32), ("num_sms", ctypes.c_int32),
                ("item_cost", ctypes.c_int32), ("unit_tokens", ctypes.c_int32),
                ("merge", ctypes.c_int32)]


class TuneResult(ctypes.Structure):
    _fields_ = [("options", PlanOptions), ("ms", ctypes.c_float)]


TUNE_IGNORE_CACHE = 1


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(LIB_PATH)
    P, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    lib.mla_decode_plan.argtypes = [P, P, i32, i32, ctypes.c_int, ctypes.c_int, i32, i32,
                                    ctypes.POINTER(P)]
    lib.mla_decode_plan_q.argtypes = [P, P, i32, i32, i32, ctypes.c_int, ctypes.c_int, i32, i32,
                                      ctypes.POINTER(P)]
    lib.mla_decode_plan_ex.argtypes = [P, P, i32, i32, i32, ctypes.c_int, ctypes.c_int, P,
                                       ctypes.POINTER(P)]
    lib.mla_decode_autotune.argtypes = [P, P, i32, i32, i32, ctypes.c_int, ctypes.c_int,
                                        P, P, P, P, P, i64, i64, P, P, sz, P, P, i32, i32, P,
                                        P, i32, ctypes.POINTER(i32), ctypes.POINTER(sz),
                                        ctypes.POINTER(P)]
    lib.mla_autotune_select.argtypes = [P, i32, i32, ctypes.POINTER(i32)]
    lib.mla_plan_workspace_size.argtypes = [P, ctypes.POINTER(sz)]
    lib.mla_plan_get_info.argtypes = [P, ctypes.POINTER(PlanInfo)]
    lib.mla_plan_get_work.argtypes = [P, P, P]
    lib.mla_plan_destroy.argtypes = [P]
    lib.mla_plan_destroy.restype = None
    lib.mla_decode_run.argtypes = [P, P, P, P, P, P, i64, i64, P, P, sz, P, P, P]
    lib.mla_decode_check.argtypes = [P, P, P]
    lib.mla_plan_set_stage1_events.argtypes = [P, P, P]
    lib.mla_decode_run_noalloc.argtypes = [P, P, P, P, P, P, i64, i64, P, P, P, P]
    lib.mla_selftest_bounded_wait.argtypes = [P, P, sz, ctypes.c_uint32, P]
    lib.mla_status_string.argtypes = [ctypes.c_int]
    lib.mla_status_string.restype = ctypes.c_char_p
    for name in ("mla_decode_plan", "mla_plan_workspace_size", "mla_plan_get_info",
                 "mla_plan_get_work", "mla_decode_run", "mla_decode_check",
                 "mla_plan_set_stage1_events", "mla_decode_run_noalloc", "mla_decode_plan_q",
                 "mla_selftest_bounded_wait", "mla_decode_plan_ex", "mla_decode_autotune",
                 "mla_autotune_select"):
        getattr(lib, name).restype = ctypes.c_int
    return lib


_lib = _load()


def mla_status_string(status: int) -> str:
    return _lib.mla_status_string(int(status)).decode()


def _check(call, status):
    if status != 0:
        raise MlaError(call, status)


def _i32_array(x):
    import numpy as np
    if x is None:
        return None, None
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    a = np.ascontiguousarray(x, dtype=np.int32)
    return a, a.ctypes.data_as(ctypes.c_void_p)


class Plan:
    """Owns an mla_plan* (host object)."""

    def __init__(self, handle, q_dtype, kv_dtype, page_size):
        self._h = handle
        self.q_dtype, self.kv_dtype, self.page_size = q_dtype, kv_dtype, page_size
        self.q_len = 1

    @property
    def handle(self):
        return self._h

    def info(self) -> PlanInfo:
        info = PlanInfo()
        _check("mla_plan_get_info", _lib.mla_plan_get_info(self._h, ctypes.byref(info)))
        return info

    @property
    def workspace_bytes(self) -> int:
        n = ctypes.c_size_t()
        _check("mla_plan_workspace_size", _lib.mla_plan_workspace_size(self._h, ctypes.byref(n)))
        return n.value

    def work(self):
        """(cta_indptr [num_ctas+1], items [num_items,4]) as numpy int32."""
        import numpy as np
        inf = self.info()
        ind = np.zeros(inf.num_ctas + 1, np.int32)
        items = np.zeros((inf.num_items, 4), np.int32)
        _check("mla_plan_get_work", _lib.mla_plan_get_work(
            self._h, ind.ctypes.data_as(ctypes.c_void_p), items.ctypes.data_as(ctypes.c_void_p)))
        return ind, items

    def set_stage1_events(self, before=None, after=None):
        """torch.cuda.Event objects (or None) recorded around each stage-1 launch."""
        b = None if before is None else ctypes.c_void_p(before.cuda_event)
        a = None if after is None else ctypes.c_void_p(after.cuda_event)
        _check("mla_plan_set_stage1_events", _lib.mla_plan_set_stage1_events(self._h, b, a))

    def __del__(self):
        if getattr(self, "_h", None):
            _lib.mla_plan_destroy(self._h)
            self._h = None


def mla_decode_plan(kv_indptr, kv_last_page_len=None, *, page_size: int, q_dtype: str,
                    kv_dtype: str, num_splits: int = 0, num_sms: int = 0,
                    batch_size: int | None = None, q_len: int = 1, item_cost: int = 0,
                    unit_tokens: int = 0, merge: int = 0) -> Plan:
    """Plan a batch from the HOST kv_indptr (in pages) and optional last-page
    lengths.  num_sms=0 queries the current CUDA device.  q_len > 1 plans
    q_len query tokens per request (mla_decode_plan_q): q, out and lse then
    hold [bs, q_len, 16, ...] rows.  item_cost / unit_tokens / merge other
    than 0 select the plan options of mla_decode_plan_ex (merge=1: always
    merge split requests with stage 2, never inside a cluster)."""
    ind, ind_p = _i32_array(kv_indptr)
    last, last_p = _i32_array(kv_last_page_len)
    bs = len(ind) - 1 if batch_size is None else int(batch_size)
    h = ctypes.c_void_p()
    if item_cost or unit_tokens or merge:
        opts = PlanOptions(int(num_splits), int(num_sms), int(item_cost), int(unit_tokens),
                           int(merge))
        _check("mla_decode_plan_ex", _lib.mla_decode_plan_ex(
            ind_p, last_p, bs, int(q_len), int(page_size), DTYPES[q_dtype], DTYPES[kv_dtype],
            ctypes.byref(opts), ctypes.byref(h)))
    elif int(q_len) == 1:
        _check("mla_decode_plan", _lib.mla_decode_plan(ind_p, last_p, bs, int(page_size),
                                                       DTYPES[q_dtype], DTYPES[kv_dtype],
                                                       int(num_splits), int(num_sms),
                                                       ctypes.byref(h)))
    else:
        _check("mla_decode_plan_q", _lib.mla_decode_plan_q(ind_p, last_p, bs, int(q_len),
                                                           int(page_size), DTYPES[q_dtype],
                                                           DTYPES[kv_dtype], int(num_splits),
                                                           int(num_sms), ctypes.byref(h)))
    plan = Plan(h, q_dtype, kv_dtype, int(page_size))
    plan.q_len = int(q_len)
    plan._keep = (ind, last)
    return plan


def _ptr(t):
    # a plain int: ctypes converts it for the void* parameter
    return None if t is None else t.data_ptr()


def _stream_ptr(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def mla_decode_run(plan: Plan, q, kv, out, *, workspace, q_scale=None, kv_scale=None,
                   kv_e8m0=None, kv_indices=None, lse=None, kv_pool_rows: int | None = None,
                   stream=None) -> None:
    """Enqueue one decode on `stream` (default: torch's current stream).

    q [bs,16,576] bf16 or uint8 (e4m3 bytes); kv [rows,576] bf16 / uint8 e4m3
    bytes, or [rows,288] uint8 packed MXFP4; out [bs,16,512] bf16; lse
    [bs,16] fp32 or None; workspace a uint8 CUDA tensor of at least
    plan.workspace_bytes; scales are fp32 CUDA tensors of one element.  With
    a plan for q_len query tokens, q, out and lse hold bs * q_len rows.
    """
    for name, t in (("q", q), ("kv", kv), ("out", out), ("workspace", workspace)):
        if t is None or not (t.is_cuda and t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    rows = kv.shape[0] if kv_pool_rows is None else int(kv_pool_rows)
    stride = 0 if kv_e8m0 is None else kv_e8m0.stride(0)
    status = _lib.mla_decode_run(plan.handle, q.data_ptr(), _ptr(q_scale), kv.data_ptr(),
                                 _ptr(kv_scale), _ptr(kv_e8m0), stride, rows, _ptr(kv_indices),
                                 workspace.data_ptr(), workspace.nbytes, out.data_ptr(),
                                 _ptr(lse), _stream_ptr(stream))
    if status:
        _check("mla_decode_run", status)


def mla_decode_run_noalloc(plan: Plan, q, kv, out, *, q_scale=None, kv_scale=None,
                           kv_e8m0=None, kv_indices=None, lse=None,
                           kv_pool_rows: int | None = None, stream=None) -> None:
    """mla_decode_run for callers that cannot allocate a workspace: the
    library's own fixed device array (16 MiB) is used instead.  Calls share
    that array, so they must not overlap on the GPU."""
    for name, t in (("q", q), ("kv", kv), ("out", out)):
        if t is None or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    rows = int(kv.shape[0]) if kv_pool_rows is None else int(kv_pool_rows)
    stride = 0 if kv_e8m0 is None else int(kv_e8m0.stride(0))
    status = _lib.mla_decode_run_noalloc(plan.handle, _ptr(q), _ptr(q_scale), _ptr(kv),
                                         _ptr(kv_scale), _ptr(kv_e8m0), stride, rows,
                                         _ptr(kv_indices), _ptr(out), _ptr(lse),
                                         _stream_ptr(stream))
    _check("mla_decode_run_noalloc", status)


def mla_decode_autotune(kv_indptr, kv_last_page_len, q, kv, out, *, page_size: int,
                        q_dtype: str, kv_dtype: str, workspace=None, q_scale=None,
                        kv_scale=None, kv_e8m0=None, kv_indices=None, lse=None,
                        kv_pool_rows: int | None = None, q_len: int = 1, reps: int = 5,
                        ignore_cache: bool = False, stream=None):
    """Time the candidate plans of this batch shape on these inputs and return
    (chosen Plan, [(options dict, median ms), ...]).  With workspace=None only
    the workspace the largest candidate needs is returned, as an int."""
    ind, ind_p = _i32_array(kv_indptr)
    last, last_p = _i32_array(kv_last_page_len)
    bs = len(ind) - 1
    results = (TuneResult * 16)()
    nres = ctypes.c_int32()
    need = ctypes.c_size_t()
    h = ctypes.c_void_p()
    rows = int(kv.shape[0]) if kv_pool_rows is None else int(kv_pool_rows)
    stride = 0 if kv_e8m0 is None else int(kv_e8m0.stride(0))
    ws_ptr = None if workspace is None else workspace.data_ptr()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("mla_decode_autotune", _lib.mla_decode_autotune(
        ind_p, last_p, bs, int(q_len), int(page_size), DTYPES[q_dtype], DTYPES[kv_dtype],
        _ptr(q), _ptr(q_scale), _ptr(kv), _ptr(kv_scale), _ptr(kv_e8m0), stride, rows,
        _ptr(kv_indices), ws_ptr, ws_bytes, _ptr(out), _ptr(lse), int(reps),
        TUNE_IGNORE_CACHE if ignore_cache else 0, _stream_ptr(stream), results, 16,
        ctypes.byref(nres), ctypes.byref(need), ctypes.byref(h)))
    if workspace is None:
        return need.value
    plan = Plan(h, q_dtype, kv_dtype, int(page_size))
    plan.q_len = int(q_len)
    table = [({"num_splits": r.options.num_splits, "num_sms": r.options.num_sms,
               "item_cost": r.options.item_cost, "unit_tokens": r.options.unit_tokens,
               "merge": r.options.merge}, r.ms)
             for r in results[: nres.value]]
    return plan, table


def mla_autotune_select(ms) -> int:
    """The autotuner's choice among candidates: ms is [candidates][reps] of
    times (negative = not run); returns the index of the smallest median."""
    import numpy as np
    a = np.ascontiguousarray(ms, dtype=np.float32)
    best = ctypes.c_int32()
    _check("mla_autotune_select", _lib.mla_autotune_select(
        a.ctypes.data_as(ctypes.c_void_p), int(a.shape[0]), int(a.shape[1]), ctypes.byref(best)))
    return best.value


def mla_selftest_bounded_wait(plan: Plan, workspace, limit_us: int = 10000, stream=None) -> None:
    """Enqueue one warp whose bounded wait on a barrier nothing arrives on runs
    out after limit_us: the next mla_decode_check raises MlaError with
    MLA_ERR_DEVICE_TIMEOUT (status 5) and clears the device error word."""
    _check("mla_selftest_bounded_wait", _lib.mla_selftest_bounded_wait(
        plan.handle, _ptr(workspace), workspace.numel() * workspace.element_size(),
        int(limit_us), _stream_ptr(stream)))


def mla_decode_check(plan: Plan, workspace=None, stream=None) -> None:
    """Synchronise, read and clear the workspace's device error word, and
    raise MlaError if it was set: status 5 (a device-side wait gave up), 1 (a
    page-table entry outside the pool), 3 (the workspace held another plan's
    table; nothing was written).  workspace=None checks the library's own
    array that mla_decode_run_noalloc uses."""
    _check("mla_decode_check", _lib.mla_decode_check(plan.handle, _ptr(workspace),
                                                     _stream_ptr(stream)))


class MlaDecoder:
    """Convenience owner of a plan and its workspace for one batch shape."""

    def __init__(self, kv_indptr, kv_last_page_len=None, *, page_size, q_dtype, kv_dtype,
                 num_splits=0, device="cuda"):
        import torch
        self.plan = mla_decode_plan(kv_indptr, kv_last_page_len, page_size=page_size,
                                    q_dtype=q_dtype, kv_dtype=kv_dtype, num_splits=num_splits)
        self.workspace = torch.empty(max(self.plan.workspace_bytes, 256), dtype=torch.uint8,
                                     device=device)

    def __call__(self, q, kv, out, **kw):
        mla_decode_run(self.plan, q, kv, out, workspace=self.workspace, **kw)
        return out
