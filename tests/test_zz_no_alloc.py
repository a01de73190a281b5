"""The allocation-free entry point, ar_allreduce_static.

Some callers cannot allocate device memory: their GPU memory is reserved in
full by another allocator, their device budget is fixed at start-up, or they
cannot afford the device-wide synchronisation of cudaMalloc / cudaFree.  For
them ar_allreduce_static runs the allreduce with every byte of device scratch
in one static array inside the library.  These tests call it through the C
ABI and check that it gives the oracle's bits and the plan path's (ar_plan_create
+ ar_execute) on two calls in a row -- the array keeps the previous call's
contents, so the second call must not depend on them -- with the status word
read back by ar_allreduce_static_check after every call and the guard bands
around every rank buffer intact; that it allocates no device memory; and that
it refuses, before any launch, a schedule whose scratch or tables exceed the
array.

The file is named to be collected last, so a run stopping at the first failure
has already run every other test.
"""

import ctypes

import pytest

import ar_synth
import collective_reduction_gb300 as ar
import oracle
from oracle.elementops import Arith

from gpu_util import RankBufs, assert_bit_equal, ensure_built, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    L = ensure_built()
    f = L.ar_allreduce_static
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_int, ctypes.c_uint64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.POINTER(ar.Params), ctypes.POINTER(ctypes.c_void_p), ctypes.c_void_p]
    c = L.ar_allreduce_static_check
    c.restype = ctypes.c_int
    c.argtypes = [ctypes.c_void_p]
    return L


def static_status(lib):
    import torch
    return ar.STATUS.get(lib.ar_allreduce_static_check(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)))


def static_call(lib, bufs, dtype, op, algo, **params):
    import torch
    p, keep = ar._params(**params)
    ptrs = (ctypes.c_void_p * len(bufs))(*[b.data_ptr() if hasattr(b, "data_ptr") else int(b) for b in bufs])
    return lib.ar_allreduce_static(len(bufs), bufs[0].numel(), ar.DTYPES[dtype], ar.OPS[op], ar.ALGOS[algo],
                                   ctypes.byref(p), ptrs, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


CASES = [
    # fused ring with ragged chunk edges (rank-streaming + element-wise kernels)
    dict(P=8, n=(1 << 20) + 3, dtype="float32", op="sum", algo="ring", params={}),
    # step form of a schedule that keeps a second partial per chunk in scratch
    dict(P=7, n=100003, dtype="float32", op="sum", algo="generalized", params={"form": "step", "r": 1}),
    # fused chains and trees over unequal groups, bf16
    dict(P=5, n=65536 + 17, dtype="bfloat16", op="sum", algo="ahc", params={"group_sizes": [2, 3]}),
    # fused DAG programs (the interpreting staged kernel)
    dict(P=7, n=200003, dtype="float32", op="max", algo="rd", params={}),
    # a fused all-gather (copy kernel), bf16
    dict(P=8, n=(1 << 18) + 5, dtype="bfloat16", op="sum", algo="ring", params={"phase": "all_gather"}),
    # a mid-sized pass of long chains (chain word kernel)
    dict(P=16, n=(1 << 18) + 1, dtype="float32", op="sum", algo="ring", params={}),
]


def run_both(lib, case, seed):
    import torch
    P, n, dtype = case["P"], case["n"], case["dtype"]
    host = ar_synth.rank_inputs(P, n, dtype, "normal", sigma=1e-2, seed=seed)
    want = oracle.run(case["algo"], host, Arith(case["op"], dtype),
                      **{k: v for k, v in case["params"].items() if k != "form"}).bufs
    a = RankBufs.from_host(host, dtype)
    b = RankBufs.from_host(host, dtype)
    plan = ar.Plan(P, n, dtype, case["op"], case["algo"], **case["params"])
    plan.execute(a.views)
    plan.check()
    plan.close()
    st = static_call(lib, b.views, dtype, case["op"], case["algo"], **case["params"])
    assert st == 0, ar.STATUS.get(st, st)
    assert static_status(lib) == "AR_OK"
    torch.cuda.synchronize()
    b.check_guards(f"static {case['algo']}")
    for r in range(P):
        got = to_host(b.views[r], dtype)
        assert_bit_equal(got, want[r], dtype, f"static vs oracle, {case['algo']} rank {r}")
        assert_bit_equal(got, to_host(a.views[r], dtype), dtype, f"static vs plan, {case['algo']} rank {r}")
    return b


def test_static_entry_matches_plan_path_on_consecutive_calls(lib):
    import torch
    # first round: every case once (the first call also does the set-up)
    for i, c in enumerate(CASES):
        run_both(lib, c, seed=i)
    # second round in reverse order: each call follows a different schedule's
    # contents in the shared array
    for i, c in reversed(list(enumerate(CASES))):
        run_both(lib, c, seed=10 + i)


def test_static_entry_allocates_no_device_memory(lib):
    import torch
    c = CASES[1]
    host = ar_synth.rank_inputs(c["P"], c["n"], c["dtype"], "normal", seed=3)
    b = RankBufs.from_host(host, c["dtype"]).views
    assert static_call(lib, b, c["dtype"], c["op"], c["algo"], **c["params"]) == 0
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(2):
        assert static_call(lib, b, c["dtype"], c["op"], c["algo"], **c["params"]) == 0
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert static_status(lib) == "AR_OK"


def test_static_entry_rejects_scratch_beyond_the_array(lib):
    import torch
    # step form, P = 7, 2^21 fp32: one scratch slot per rank = 7 x 8 MiB
    # = 56 MiB > the array's slot area; refused before any launch
    P, n = 7, 1 << 21
    b = [torch.zeros(n, dtype=torch.float32, device="cuda") for _ in range(P)]
    st = static_call(lib, b, "float32", "sum", "generalized", form="step", r=1)
    assert ar.STATUS[st] == "AR_ERR_UNSUPPORTED"
    for t in b:
        assert int(torch.count_nonzero(t)) == 0


def test_static_entry_rejects_tables_beyond_the_array(lib):
    import torch
    # the step form of a pipelined chain with 4096 blocks over 16 ranks:
    # about 120 000 work items, some 2 MB of tables > AR_STATIC_TABLE_BYTES
    P, n = 16, 1 << 17
    assert ar.Schedule(P, n, "float32", "sum", "pipeline", blocks=4096, form="step").lowering()["items"] * 16 \
        > (1 << 20)
    b = [torch.zeros(n, dtype=torch.float32, device="cuda") for _ in range(P)]
    st = static_call(lib, b, "float32", "sum", "pipeline", blocks=4096, form="step")
    assert ar.STATUS[st] == "AR_ERR_UNSUPPORTED"
    torch.cuda.synchronize()
    for t in b:
        assert int(torch.count_nonzero(t)) == 0

