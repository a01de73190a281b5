"""Single-GPU allreduce schedule engine for GB300 (sm_103a): Python binding.

This module only marshals arguments to the C ABI of ``libar.so`` (declared in
``include/ar.h``); every step of the allreduce runs in the library's CUDA
kernels.  There is no CPU fallback: if the library is not built, every call
raises.

    import torch, collective_reduction_gb300 as ar
    bufs = [torch.randn(1 << 20, device="cuda") for _ in range(8)]
    plan = ar.Plan(8, 1 << 20, "float32", "sum", "ring")
    plan.execute(bufs)            # every buffer now holds the sum
"""

import ctypes
import os

DTYPES = {"int32": 0, "float32": 1, "bfloat16": 2}
OPS = {"sum": 0, "prod": 1, "max": 2, "min": 3, "avg": 4}
ALGOS = {"ring": 0, "binomial": 1, "rh": 2, "rd": 3, "hybrid": 4, "generalized": 5, "ahc": 6, "pipeline": 7}
FORMS = {"fused": 0, "step": 1}
ORDERS = {"faithful": 0, "fp32acc": 1}
GROUPS = {"cyclic": 0, "xor": 1}
PHASES = {"allreduce": 0, "reduce_scatter": 1, "all_gather": 2}
JIT = {"auto": 0, "on": 1, "off": -1}
ESIZE = {"int32": 4, "float32": 4, "bfloat16": 2}
KERNEL_STREAM, KERNEL_STAGED, KERNEL_ELEMENTWISE, KERNEL_DAG_JIT, KERNEL_WORD_JIT, KERNEL_CHAIN_WORD = 1, 2, 4, 8, 16, 32
KERNEL_COPY, KERNEL_FEW = 64, 128
MAX_RANKS = 64

STATUS = {0: "AR_OK", 1: "AR_ERR_INVALID_ARG", 2: "AR_ERR_UNSUPPORTED", 3: "AR_ERR_CUDA",
          4: "AR_ERR_NOMEM", 5: "AR_ERR_TIMEOUT", 6: "AR_ERR_INTERNAL"}

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libar.so")


class ArError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        self.name = STATUS.get(status, str(status))
        super().__init__(f"{where}: {self.name} ({_status_text(status)})")


class Params(ctypes.Structure):
    _fields_ = [("form", ctypes.c_int), ("order", ctypes.c_int), ("group", ctypes.c_int),
                ("r", ctypes.c_int), ("k1", ctypes.c_int), ("n_groups", ctypes.c_int),
                ("group_sizes", ctypes.POINTER(ctypes.c_int)), ("blocks", ctypes.c_int),
                ("phase", ctypes.c_int), ("jit", ctypes.c_int)]


class Info(ctypes.Structure):
    _fields_ = [("P", ctypes.c_int), ("dtype", ctypes.c_int), ("op", ctypes.c_int), ("algo", ctypes.c_int),
                ("form", ctypes.c_int), ("order", ctypes.c_int), ("phase", ctypes.c_int), ("n", ctypes.c_uint64),
                ("steps", ctypes.c_int), ("sent_bytes_max", ctypes.c_uint64),
                ("sent_bytes_total", ctypes.c_uint64), ("combines", ctypes.c_uint64),
                ("max_slots", ctypes.c_int), ("n_segments", ctypes.c_int),
                ("hbm_bytes", ctypes.c_uint64), ("scratch_bytes", ctypes.c_uint64),
                ("launches", ctypes.c_int), ("tile_bytes", ctypes.c_int), ("n_programs", ctypes.c_int),
                ("n_items", ctypes.c_uint64), ("kernels", ctypes.c_int), ("messages", ctypes.c_uint64)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}


class LoweringInfo(ctypes.Structure):
    _fields_ = [("items", ctypes.c_uint64), ("launch_sets", ctypes.c_int), ("windows", ctypes.c_int),
                ("tiling_ok", ctypes.c_int), ("windows_ok", ctypes.c_int), ("wave_balance", ctypes.c_double),
                ("stream_tile_bytes", ctypes.c_int), ("stream_stages", ctypes.c_int),
                ("staged_tile_bytes", ctypes.c_int), ("staged_stages", ctypes.c_int), ("dag_words", ctypes.c_uint64),
                ("word_sets", ctypes.c_int), ("word_kernel_words", ctypes.c_uint64), ("stream_tmem", ctypes.c_int),
                ("copy_sets", ctypes.c_int), ("few_sets", ctypes.c_int)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}


class CostModel(ctypes.Structure):
    """Step-form cost: alpha per round, beta per byte sent, gamma per byte
    combined and delta per message, summed over all ranks."""
    _fields_ = [("alpha_us", ctypes.c_double), ("beta_us_per_byte", ctypes.c_double),
                ("gamma_us_per_byte", ctypes.c_double), ("delta_us_per_message", ctypes.c_double)]


_lib = None
_VP = ctypes.c_void_p
_EXPORTS = {
    "ar_schedule_create": (ctypes.c_int, [ctypes.c_int, ctypes.c_uint64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          ctypes.POINTER(Params), ctypes.POINTER(_VP)]),
    "ar_schedule_destroy": (ctypes.c_int, [_VP]),
    "ar_schedule_query": (ctypes.c_int, [_VP, ctypes.POINTER(Info)]),
    "ar_schedule_step_sent": (ctypes.c_int, [_VP, ctypes.c_int, ctypes.POINTER(ctypes.c_uint64)]),
    "ar_schedule_tree": (ctypes.c_int, [_VP, ctypes.c_int, ctypes.c_uint64, ctypes.c_char_p, ctypes.c_size_t,
                                        ctypes.POINTER(ctypes.c_size_t)]),
    "ar_plan_create": (ctypes.c_int, [ctypes.c_int, ctypes.c_uint64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                      ctypes.POINTER(Params), ctypes.POINTER(_VP)]),
    "ar_plan_destroy": (ctypes.c_int, [_VP]),
    "ar_plan_query": (ctypes.c_int, [_VP, ctypes.POINTER(Info)]),
    "ar_execute": (ctypes.c_int, [_VP, ctypes.POINTER(_VP), _VP]),
    "ar_execute_host": (ctypes.c_int, [_VP, ctypes.POINTER(_VP), ctypes.POINTER(_VP), _VP]),
    "ar_plan_check": (ctypes.c_int, [_VP]),
    "ar_plan_check_buffers": (ctypes.c_int, [_VP, ctypes.POINTER(_VP)]),
    "ar_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "ar_schedule_dag_kernel": (ctypes.c_int, [_VP, ctypes.POINTER(ctypes.c_size_t)]),
    "ar_schedule_lowering": (ctypes.c_int, [_VP, ctypes.POINTER(LoweringInfo)]),
    "ar_selftest_bounded_wait": (ctypes.c_int, [ctypes.c_uint32, _VP]),
    "ar_cost_model_default": (ctypes.c_int, [ctypes.POINTER(CostModel)]),
    "ar_cost_predict": (ctypes.c_int, [_VP, ctypes.POINTER(CostModel), ctypes.POINTER(ctypes.c_double)]),
    "ar_cost_optimal_r": (ctypes.c_int, [ctypes.c_int, ctypes.c_uint64, ctypes.POINTER(CostModel),
                                         ctypes.POINTER(ctypes.c_int)]),
    "ar_cost_select": (ctypes.c_int, [ctypes.c_int, ctypes.c_uint64, ctypes.c_int, ctypes.c_int,
                                      ctypes.POINTER(CostModel), ctypes.POINTER(ctypes.c_int),
                                      ctypes.POINTER(Params), ctypes.POINTER(ctypes.c_double)]),
}


def lib():
    """The loaded libar.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run `python -m collective_reduction_gb300.build` "
                               "(the engine has no non-CUDA fallback)")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _EXPORTS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _status_text(s):
    try:
        return lib().ar_status_string(s).decode()
    except Exception:  # the library itself may be what is missing
        return STATUS.get(s, "unknown")


def _check(status, where):
    if status != 0:
        raise ArError(status, where)


def _params(form="fused", order="faithful", group="cyclic", r=0, k1=0, group_sizes=None, blocks=1,
            phase="allreduce", jit="auto"):
    p = Params(FORMS[form], ORDERS[order], GROUPS[group], int(r), int(k1), 0, None, int(blocks), PHASES[phase],
               JIT[jit])
    keep = None
    if group_sizes is not None:
        keep = (ctypes.c_int * len(group_sizes))(*[int(g) for g in group_sizes])
        p.n_groups = len(group_sizes)
        p.group_sizes = keep
    return p, keep


def _ptrs(bufs):
    out = (_VP * len(bufs))()
    for i, b in enumerate(bufs):
        out[i] = b.data_ptr() if hasattr(b, "data_ptr") else int(b)
    return out


def _stream_handle(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if hasattr(stream, "cuda_stream"):
        return stream.cuda_stream
    return int(stream)


class Schedule:
    """Host-only compiled schedule: counters, per-round traffic, trees."""

    def __init__(self, P, n, dtype, op, algo, **params):
        self.P, self.n = P, n
        p, self._keep = _params(**params)
        h = _VP()
        _check(lib().ar_schedule_create(P, n, DTYPES[dtype], OPS[op], ALGOS[algo], ctypes.byref(p),
                                        ctypes.byref(h)), "ar_schedule_create")
        self._h = h

    def info(self):
        i = Info()
        _check(lib().ar_schedule_query(self._h, ctypes.byref(i)), "ar_schedule_query")
        return i.as_dict()

    def step_sent(self, step):
        out = (ctypes.c_uint64 * self.P)()
        _check(lib().ar_schedule_step_sent(self._h, step, out), "ar_schedule_step_sent")
        return list(out)

    def tree(self, rank, elem):
        need = ctypes.c_size_t(0)
        lib().ar_schedule_tree(self._h, rank, elem, None, 0, ctypes.byref(need))
        buf = ctypes.create_string_buffer(max(1, need.value))
        _check(lib().ar_schedule_tree(self._h, rank, elem, buf, need.value, ctypes.byref(need)),
               "ar_schedule_tree")
        return buf.value.decode()

    def dag_kernel_bytes(self):
        """Code size of the run-time DAG kernel a plan of this schedule would
        compile (0: no DAG program on the staged kernel); compiles on the host."""
        n = ctypes.c_size_t(0)
        _check(lib().ar_schedule_dag_kernel(self._h, ctypes.byref(n)), "ar_schedule_dag_kernel")
        return n.value

    def lowering(self):
        """The work items a plan of this schedule would launch, with the host
        checks of their tiling and host-path windows (ar_schedule_lowering)."""
        info = LoweringInfo()
        _check(lib().ar_schedule_lowering(self._h, ctypes.byref(info)), "ar_schedule_lowering")
        return info.as_dict()

    def close(self):
        if getattr(self, "_h", None):
            lib().ar_schedule_destroy(self._h)
            self._h = None

    __del__ = close


class Plan:
    """A compiled, uploaded allreduce for P buffers of n elements on the
    current CUDA device."""

    def __init__(self, P, n, dtype, op, algo, **params):
        self.P, self.n, self.dtype = P, n, dtype
        p, self._keep = _params(**params)
        h = _VP()
        _check(lib().ar_plan_create(P, n, DTYPES[dtype], OPS[op], ALGOS[algo], ctypes.byref(p),
                                    ctypes.byref(h)), "ar_plan_create")
        self._h = h

    def info(self):
        i = Info()
        _check(lib().ar_plan_query(self._h, ctypes.byref(i)), "ar_plan_query")
        return i.as_dict()

    def execute(self, bufs, stream=None):
        """Enqueue the allreduce over P device buffers (tensors or raw device
        addresses) on `stream` (default: torch's current stream)."""
        if len(bufs) != self.P:
            raise ValueError(f"expected {self.P} buffers, got {len(bufs)}")
        _check(lib().ar_execute(self._h, _ptrs(bufs), _VP(_stream_handle(stream))), "ar_execute")

    def execute_host(self, host_bufs, dev_bufs, stream=None):
        """Copy host buffers in, allreduce, copy every result back, sync."""
        _check(lib().ar_execute_host(self._h, _ptrs(host_bufs), _ptrs(dev_bufs), _VP(_stream_handle(stream))),
               "ar_execute_host")

    def check(self):
        """Synchronise; raise ArError(AR_ERR_TIMEOUT) if a kernel gave up a wait,
        ArError(AR_ERR_INTERNAL) if a kernel met a program it does not run or
        wrote past the plan's scratch."""
        _check(lib().ar_plan_check(self._h), "ar_plan_check")

    def check_buffers(self, bufs):
        """The status ar_execute's buffer checks give these P buffers (residency
        on the plan's device, extent, alignment, overlap); launches nothing."""
        if len(bufs) != self.P:
            raise ValueError(f"expected {self.P} buffers, got {len(bufs)}")
        return STATUS.get(lib().ar_plan_check_buffers(self._h, _ptrs(bufs)), "unknown")

    def close(self):
        if getattr(self, "_h", None):
            lib().ar_plan_destroy(self._h)
            self._h = None

    __del__ = close


# ---------------------------------------------------------------- cost model

def cost_model(alpha_us=None, beta_us_per_byte=None, gamma_us_per_byte=None):
    """The fitted GB300 step-form model, with any field overridden."""
    m = CostModel()
    _check(lib().ar_cost_model_default(ctypes.byref(m)), "ar_cost_model_default")
    if alpha_us is not None:
        m.alpha_us = alpha_us
    if beta_us_per_byte is not None:
        m.beta_us_per_byte = beta_us_per_byte
    if gamma_us_per_byte is not None:
        m.gamma_us_per_byte = gamma_us_per_byte
    return m


def cost_predict(schedule, model=None):
    """Predicted step-form microseconds of a Schedule."""
    model = model or cost_model()
    us = ctypes.c_double()
    _check(lib().ar_cost_predict(schedule._h, ctypes.byref(model), ctypes.byref(us)), "ar_cost_predict")
    return us.value


def optimal_r(P, bytes_per_rank, model=None):
    """Removed distribution steps minimising the generalized schedule's cost
    ("A Generalization of the Allreduce Operation", eq. 37), in 0..L-1."""
    model = model or cost_model()
    r = ctypes.c_int()
    _check(lib().ar_cost_optimal_r(P, bytes_per_rank, ctypes.byref(model), ctypes.byref(r)), "ar_cost_optimal_r")
    return r.value


def select(P, n, dtype, op, model=None):
    """(algo, params, predicted microseconds) of the cheapest step-form
    schedule under the model; params fit Plan(..., **params)."""
    model = model or cost_model()
    algo = ctypes.c_int()
    p = Params()
    us = ctypes.c_double()
    _check(lib().ar_cost_select(P, n, DTYPES[dtype], OPS[op], ctypes.byref(model), ctypes.byref(algo),
                                ctypes.byref(p), ctypes.byref(us)), "ar_cost_select")
    name = {v: k for k, v in ALGOS.items()}[algo.value]
    params = {"form": "step", "order": "faithful", "group": "cyclic", "r": p.r, "k1": p.k1}
    return name, params, us.value


def selftest_bounded_wait(timeout_ms=100, stream=None):
    """Runs the bounded-wait self-test; returns the status name ("AR_ERR_TIMEOUT"
    when the wait gave up as designed)."""
    st = lib().ar_selftest_bounded_wait(int(timeout_ms), _VP(_stream_handle(stream)))
    return STATUS.get(st, str(st))
