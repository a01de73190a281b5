"""Host-side tests of the C ABI (no GPU): the library loads and exports every
function ``include/ar.h`` declares, and the schedule compiler behind
``ar_schedule_*`` builds exactly the reduction trees and per-round traffic of
the oracle's independent simulation."""

import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from oracle.chunking import ceil_log2
from oracle.elementops import Symbolic, leaf_buffers, tree_str

ar = pytest.importorskip("collective_reduction_gb300")
HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "ar.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(ar.LIB_PATH):
        from collective_reduction_gb300 import build
        build.build()
    return ar.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ar_[a-z_]+)\s*\(", text)))


def test_header_declares_the_abi():
    names = declared_functions()
    for must in ("ar_plan_create", "ar_execute", "ar_plan_destroy", "ar_plan_query", "ar_status_string",
                 "ar_schedule_create", "ar_schedule_tree", "ar_execute_host", "ar_plan_check"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for s in range(7):
        assert lib.ar_status_string(s).decode().startswith(ar.STATUS[s])
    assert lib.ar_status_string(99)


def _cases():
    for P in (1, 2, 3, 4, 5, 7, 8, 12, 16):
        L = ceil_log2(P)
        Lp = ceil_log2(1 << (P.bit_length() - 1))
        yield "ring", P, {}
        yield "binomial", P, {}
        for r in range(L + 1):
            yield "generalized", P, {"group": "cyclic", "r": r}
        yield "rd", P, {}
        yield "rh", P, {}
        for k1 in range(Lp + 1):
            yield "hybrid", P, {"k1": k1}
        if P & (P - 1) == 0:
            for r in range(L + 1):
                yield "generalized", P, {"group": "xor", "r": r}
        for sizes in ([P], [1] * P, [P // 2, P - P // 2] if P > 1 else [1], [2, P - 2] if P >= 4 else [P]):
            yield "ahc", P, {"group_sizes": sizes}
        for m in (1, 3):
            yield "pipeline", P, {"blocks": m}


@pytest.mark.parametrize("op", ["max", "sum"])
def test_compiler_trees_and_traffic_match_oracle(lib, op):
    for algo, P, kw in _cases():
        for n in (2 * P + 3, P - 1 if P > 1 else 1):
            s = ar.Schedule(P, n, "float32", op, algo, **kw)
            res = oracle.run(algo, leaf_buffers(P, n), Symbolic(), **kw)
            info = s.info()
            assert info["steps"] == res.steps, (algo, P, kw)
            for i in range(res.steps):
                assert s.step_sent(i) == res.sent[i], (algo, P, kw, i)
            for r in range(P):
                for e in range(n):
                    assert s.tree(r, e) == tree_str(res.bufs[r][e]), (algo, P, kw, r, e)
            assert info["combines"] == res.combines, (algo, P, kw)
            s.close()


def test_compiler_counters_large_P(lib):
    # P = 64 ring and P = 63 generalized: steps and traffic closed forms
    s = ar.Schedule(64, 64 * 1000, "float32", "sum", "ring")
    i = s.info()
    assert i["steps"] == 126 and i["sent_bytes_max"] == 2 * 63 * 1000 * 4
    g = ar.Schedule(63, 63 * 10, "float32", "sum", "generalized", r=3)
    assert g.info()["steps"] == 2 * 6 - 3
    assert g.info()["max_slots"] == 2


def test_ahc_twelve_chunks(lib):
    s = ar.Schedule(5, 24, "bfloat16", "sum", "ahc", group_sizes=[2, 3])
    i = s.info()
    assert i["steps"] == 6
    # 12 chunks of 2 elements; segments split at chunk boundaries only
    assert i["n_segments"] == 12


@pytest.mark.parametrize("args,status", [
    ((0, 8, "float32", "sum", "ring", {}), "AR_ERR_INVALID_ARG"),
    ((65, 8, "float32", "sum", "ring", {}), "AR_ERR_UNSUPPORTED"),
    ((6, 8, "float32", "sum", "hybrid", {"k1": 3}), "AR_ERR_INVALID_ARG"),
    ((8, 8, "float32", "sum", "hybrid", {"k1": 4}), "AR_ERR_INVALID_ARG"),
    ((8, 8, "float32", "sum", "hybrid", {"k1": -1}), "AR_ERR_INVALID_ARG"),
    ((12, 8, "float32", "sum", "generalized", {"group": "xor"}), "AR_ERR_UNSUPPORTED"),
    ((7, 8, "float32", "sum", "generalized", {"r": 4}), "AR_ERR_INVALID_ARG"),
    ((5, 8, "float32", "sum", "ahc", {"group_sizes": [2, 2]}), "AR_ERR_INVALID_ARG"),
    ((5, 8, "float32", "sum", "ahc", {"group_sizes": [0, 5]}), "AR_ERR_INVALID_ARG"),
    ((5, 8, "float32", "sum", "ahc", {}), "AR_ERR_INVALID_ARG"),
    ((5, 8, "float32", "sum", "ring", {"form": "step", "order": "fp32acc"}), "AR_ERR_UNSUPPORTED"),
    ((5, 8, "float32", "sum", "pipeline", {"blocks": -1}), "AR_ERR_INVALID_ARG"),
    ((5, 8, "float32", "sum", "pipeline", {"blocks": 4097}), "AR_ERR_INVALID_ARG"),
    ((60, 8, "float32", "sum", "ahc", {"group_sizes": [7, 8, 9, 11, 13, 12]}), "AR_ERR_UNSUPPORTED"),
])
def test_invalid_requests_rejected(lib, args, status):
    P, n, dt, op, algo, kw = args
    with pytest.raises(ar.ArError) as e:
        ar.Schedule(P, n, dt, op, algo, **kw)
    assert e.value.name == status


def test_raw_abi_null_checks(lib):
    assert lib.ar_schedule_create(4, 8, 1, 0, 0, None, None) == 1
    assert lib.ar_schedule_query(None, None) == 1
    assert lib.ar_execute(None, None, None) == 1
    assert lib.ar_plan_query(None, None) == 1
    assert lib.ar_plan_destroy(None) == 1
    assert lib.ar_plan_check(None) == 1
    bad_dtype = ctypes.c_void_p()
    assert lib.ar_schedule_create(4, 8, 7, 0, 0, None, ctypes.byref(bad_dtype)) == 1
    assert lib.ar_schedule_create(4, 8, 1, 9, 0, None, ctypes.byref(bad_dtype)) == 1
    assert lib.ar_schedule_create(4, 8, 1, 0, 42, None, ctypes.byref(bad_dtype)) == 1


def test_tree_buffer_too_small(lib):
    s = ar.Schedule(4, 8, "float32", "sum", "ring")
    need = ctypes.c_size_t(0)
    buf = ctypes.create_string_buffer(2)
    assert lib.ar_schedule_tree(s._h, 0, 0, buf, 2, ctypes.byref(need)) == 1
    assert need.value == len("(3+(2+(1+0)))") + 1
    assert lib.ar_schedule_tree(s._h, 4, 0, buf, 2, ctypes.byref(need)) == 1
    assert lib.ar_schedule_tree(s._h, 0, 8, buf, 2, ctypes.byref(need)) == 1


def _split_cases():
    for P in (1, 2, 3, 5, 7, 8, 12, 16):
        yield "ring", P, {}
        yield "rh", P, {}
        yield "generalized", P, {"group": "cyclic"}
        if P & (P - 1) == 0:
            yield "generalized", P, {"group": "xor"}


@pytest.mark.parametrize("phase", ["reduce_scatter", "all_gather"])
def test_compiler_halves_match_oracle(lib, phase):
    """The reduce-scatter / all-gather plans: rounds, traffic and, on every
    element the half defines, the tree, as in the oracle's simulation."""
    for algo, P, kw in _split_cases():
        for n in (2 * P + 3, P - 1 if P > 1 else 1):
            s = ar.Schedule(P, n, "float32", "sum", algo, phase=phase, **kw)
            res = oracle.run(algo, leaf_buffers(P, n), Symbolic(), phase=phase, **kw)
            info = s.info()
            assert info["phase"] == ar.PHASES[phase]
            assert info["steps"] == res.steps, (algo, P, kw)
            for i in range(res.steps):
                assert s.step_sent(i) == res.sent[i], (algo, P, kw, i)
            assert info["combines"] == res.combines
            if phase == "reduce_scatter":
                cells = [(rank, e) for rank, lo, hi in res.info["owner"] for e in range(lo, hi)]
            else:
                cells = [(rank, e) for rank in range(P) for e in range(n)]
            for rank, e in cells:
                assert s.tree(rank, e) == tree_str(res.bufs[rank][e]), (algo, P, kw, rank, e)
            s.close()


@pytest.mark.parametrize("algo,kw,status", [
    ("binomial", {}, "AR_ERR_UNSUPPORTED"),
    ("rd", {}, "AR_ERR_UNSUPPORTED"),
    ("hybrid", {"k1": 1}, "AR_ERR_UNSUPPORTED"),
    ("generalized", {"r": 1}, "AR_ERR_UNSUPPORTED"),
    ("ahc", {"group_sizes": [3, 5]}, "AR_ERR_UNSUPPORTED"),
    ("pipeline", {"blocks": 2}, "AR_ERR_UNSUPPORTED"),
])
def test_halves_rejected_for_other_schedules(lib, algo, kw, status):
    for phase in ("reduce_scatter", "all_gather"):
        with pytest.raises(ar.ArError) as e:
            ar.Schedule(8, 64, "float32", "sum", algo, phase=phase, **kw)
        assert e.value.name == status


def test_halves_parameter_checks(lib):
    with pytest.raises(ar.ArError) as e:
        ar.Schedule(8, 64, "float32", "sum", "ring", phase="all_gather", order="fp32acc")
    assert e.value.name == "AR_ERR_UNSUPPORTED"
    p, _keep = ar._params()
    p.phase = 3
    h = ctypes.c_void_p()
    assert lib.ar_schedule_create(8, 64, 1, 0, 0, ctypes.byref(p), ctypes.byref(h)) == 1
    # the fp32-accumulation reduce-scatter is a one-pass plan too
    s = ar.Schedule(8, 64, "bfloat16", "sum", "ring", phase="reduce_scatter", order="fp32acc")
    assert s.info()["steps"] == 7


def test_avg_requests(lib):
    with pytest.raises(ar.ArError) as e:
        ar.Schedule(4, 64, "int32", "avg", "ring")
    assert e.value.name == "AR_ERR_UNSUPPORTED"
    h = ctypes.c_void_p()
    assert lib.ar_schedule_create(4, 64, 1, 5, 0, None, ctypes.byref(h)) == 1
    # avg keeps the sum's trees and counters
    for algo, kw in (("ring", {}), ("generalized", {"r": 2}), ("binomial", {}), ("rh", {"phase": "reduce_scatter"})):
        a = ar.Schedule(7, 40, "float32", "avg", algo, **kw).info()
        s = ar.Schedule(7, 40, "float32", "sum", algo, **kw).info()
        for k in ("steps", "combines", "sent_bytes_max", "sent_bytes_total", "n_segments"):
            assert a[k] == s[k], (algo, k)


@pytest.mark.parametrize("algo,P,op,kw", [
    ("generalized", 7, "sum", {"r": 1}), ("generalized", 7, "sum", {"r": 3}), ("rd", 8, "max", {}),
    ("generalized", 12, "min", {"r": 2}), ("generalized", 7, "avg", {"r": 2}),
])
@pytest.mark.parametrize("dtype", ["int32", "float32", "bfloat16"])
def test_dag_kernel_compiles_on_the_host(lib, algo, P, op, kw, dtype):
    """The run-time DAG kernel of a plan with rank-specific programs compiles
    for sm_103a (NVRTC, no GPU needed)."""
    if op == "avg" and dtype == "int32":
        pytest.skip("avg has no integer form")
    s = ar.Schedule(P, P * 4096, dtype, op, algo, **kw)
    try:
        nbytes = s.dag_kernel_bytes()
    except ar.ArError as e:
        if e.name == "AR_ERR_UNSUPPORTED":
            pytest.skip("NVRTC is not available on this host")
        raise
    if dtype == "int32" and algo == "rd":
        assert nbytes == 0  # every int32 op commutes: one shared tree, no DAG program
    else:
        assert nbytes > 0


def test_no_dag_kernel_for_streaming_plans(lib):
    for algo, kw in (("ring", {}), ("rh", {}), ("binomial", {}), ("generalized", {"r": 2})):
        # sum trees are shared by every rank: no DAG program, nothing to compile
        assert ar.Schedule(8, 8 * 4096, "float32", "sum", algo, **kw).dag_kernel_bytes() == 0
    # the step form's cyclic rounds are versioned into independent chains
    for P, r in ((7, 3), (12, 4), (31, 5)):
        s = ar.Schedule(P, P * 4096, "float32", "max", "generalized", r=r, form="step")
        assert s.dag_kernel_bytes() == 0, (P, r)


def test_jit_parameter_checked(lib):
    p, _keep = ar._params()
    p.jit = 2
    h = ctypes.c_void_p()
    assert lib.ar_schedule_create(8, 64, 1, 0, 0, ctypes.byref(p), ctypes.byref(h)) == 1


def test_selftest_timeout_range_checked_on_host(lib):
    assert lib.ar_selftest_bounded_wait(0, None) == 1
    assert lib.ar_selftest_bounded_wait(10001, None) == 1


# ---- the lowering: work items and host-path windows -----------------------------------

def _random_plans(count, seed):
    rng = np.random.default_rng(seed)
    algos = ["ring", "binomial", "rh", "rd", "hybrid", "generalized", "ahc", "pipeline"]
    out = []
    while len(out) < count:
        P = int(rng.choice([2, 3, 4, 5, 7, 8, 12, 13, 16, 31, 32, 63, 64]))
        n = int(rng.choice([rng.integers(1, 5000), rng.integers(1 << 18, 1 << 22), rng.integers(1 << 22, 1 << 25)]))
        algo = str(rng.choice(algos))
        dtype = str(rng.choice(["int32", "float32", "bfloat16"]))
        kw = {"form": str(rng.choice(["fused", "step"]))}
        if algo == "generalized":
            kw["r"] = int(rng.integers(0, ceil_log2(P) + 1))
        if algo == "hybrid":
            kw["k1"] = int(rng.integers(0, ceil_log2(P) + 1))
        if algo == "ahc":
            kw["group_sizes"] = [P // 2, P - P // 2] if P >= 4 else [P]
        if algo == "pipeline":
            kw["blocks"] = int(rng.integers(1, 9))
        if kw["form"] == "fused" and rng.random() < 0.3:
            kw["order"] = "fp32acc"
        try:
            s = ar.Schedule(P, n, dtype, "sum", algo, **kw)
        except RuntimeError:
            continue  # a combination the compiler rejects (e.g. RH at P != 2^k)
        out.append(((P, n, dtype, algo, kw), s))
    return out


def test_lowering_tiles_every_range_and_windows_hold_their_items(lib):
    """For random plans (sizes from a few elements to 2^25, every schedule,
    both forms), the work items the kernels would run cover every element
    range exactly once per program, and the host path's windows are
    consecutive and contain their items — checked by code apart from the
    lowering."""
    for args, s in _random_plans(160, seed=11):
        low = s.lowering()
        assert low["tiling_ok"] == 1, args
        assert low["windows_ok"] == 1, args
        assert low["wave_balance"] >= 1.0
        s.close()


def test_wave_balance_closed_form(lib):
    """Round robin over 152 CTAs: P = 64 x 2^23 fp32 RH (single trees of 64
    leaves, rank-streaming kernel) has 64 chunks of 2^17 elements, 16 whole
    32 KB tiles each, 1024 equal items: 112 CTAs take 7 and 40 take 6, so the
    largest share over the mean is 7 / (1024 / 152).
    P = 16 x 2^25 RH (single trees of 16 leaves) has 4096 items: 27 / (4096 /
    152).  P = 8 x 2^26 runs on the few-input kernel, a CTA per 16 KB item
    (16384), for the ring's chains and RH's trees alike.  Windows: 2 GiB of
    rank data makes 16 windows of 128 MB."""
    low = ar.Schedule(64, 1 << 23, "float32", "sum", "rh").lowering()
    assert low["items"] == 1024 and low["windows"] == 16
    assert abs(low["wave_balance"] - 7 / (1024 / 152)) < 1e-9
    low = ar.Schedule(16, 1 << 25, "float32", "sum", "rh").lowering()
    assert low["items"] == 4096 and low["windows"] == 16 and low["few_sets"] == 0
    assert abs(low["wave_balance"] - 27 / (4096 / 152)) < 1e-9
    for algo in ("ring", "rh"):
        low = ar.Schedule(8, 1 << 26, "float32", "sum", algo).lowering()
        assert low["items"] == 16384 and low["few_sets"] == 1 and low["windows"] == 16


def test_stream_geometry_follows_the_programs(lib):
    """Pipeline depth and rank tile of the rank-streaming kernel as the
    lowering picks them: 3 stages of 32 KB for chains over 4-byte elements
    (the step form's rounds), 4 for bf16 chains, trees of more than 8 leaves
    with their stack in tensor memory on 4 stages of 32 KB, bf16 fp32
    accumulation on 7 of 24 KB.  Fused chains and fp32 accumulations of up to
    16 inputs, of more in sets of at least 1.5 GiB, and trees of up to 8
    leaves run on the few-input kernel instead."""
    def low(P, dtype, algo, op="sum", **kw):
        return ar.Schedule(P, P * (1 << 16), dtype, op, algo, **kw).lowering()
    geo = lambda *x, **kw: (low(*x, **kw)["stream_tile_bytes"], low(*x, **kw)["stream_stages"])
    assert geo(32, "float32", "ring", form="step") == (32768, 3)
    assert geo(32, "int32", "ring", form="step") == (32768, 3)
    assert geo(32, "bfloat16", "ring", form="step") == (32768, 4)
    assert geo(16, "float32", "rh") == (32768, 4)       # 4 stack entries in tensor memory
    assert geo(64, "float32", "rh") == (32768, 4)       # 6 stack entries in tensor memory
    assert geo(32, "bfloat16", "binomial") == (32768, 4)
    tm = lambda P, algo: low(P, "float32", algo)["stream_tmem"]
    assert tm(64, "rh") == 1 and tm(32, "binomial") == 1 and tm(16, "rh") == 1
    assert tm(8, "rh") == 0 and tm(8, "ring") == 0
    for P, dtype in ((8, "bfloat16"), (16, "float32"), (2, "bfloat16")):
        assert low(P, dtype, "ring", order="fp32acc")["few_sets"] == 1
    # 64 inputs below 1.5 GiB of traffic (8 MiB of bf16 per rank): the
    # rank-streaming kernel, fp32 accumulation on 7 stages of 24 KB, chains
    # on 4 of 32 KB
    assert geo(64, "bfloat16", "ring", order="fp32acc") == (24576, 7)
    assert geo(64, "bfloat16", "ring") == (32768, 4)
    big = ar.Schedule(64, 1 << 24, "float32", "sum", "ring").lowering()
    assert big["few_sets"] == 1 and big["tiling_ok"] == 1


@pytest.mark.parametrize("P,algo,kw", [(31, "generalized", {"r": 5}), (64, "rd", {}), (13, "generalized", {"r": 2})])
def test_compiled_dag_lowering(lib, P, algo, kw):
    """Plans whose DAG programs will be compiled (NVRTC present, jit on) are
    lowered without the interpreter's shared-memory temporaries; programs of
    17 to 32 inputs get tiles of whole 1 KB units (one 32-bit word per
    consumer thread), programs of more go to the word kernel.  The items tile
    every range either way, and the generated kernel compiles."""
    n = (1 << 20) + 37
    s = ar.Schedule(P, n, "float32", "max", algo, jit="on", **kw)
    low = s.lowering()
    off = ar.Schedule(P, n, "float32", "max", algo, jit="off", **kw).lowering()
    assert low["tiling_ok"] == 1 and off["tiling_ok"] == 1
    assert off["dag_words"] > 0 and off["word_sets"] == 0
    if s.dag_kernel_bytes() == 0:
        pytest.skip("NVRTC is not available on this host")
    if P > 32:  # the word kernel: every input word of a position in registers
        assert low["word_sets"] == 1 and low["word_kernel_words"] > 0 and low["dag_words"] == 0
        return
    assert low["dag_words"] > 0 and low["word_sets"] == 0
    if P > 16:
        assert low["staged_tile_bytes"] % 1024 == 0 and low["staged_stages"] >= 3
    assert low["staged_tile_bytes"] * low["staged_stages"] >= off["staged_tile_bytes"] * off["staged_stages"]


@pytest.mark.parametrize("op,dtype,word", [("max", "bfloat16", True), ("min", "bfloat16", True),
                                           ("sum", "bfloat16", False), ("max", "float32", False)])
def test_bf16_select_programs_go_to_the_word_kernel_from_25_inputs(lib, op, dtype, word):
    """bf16 max / min programs of 25 to 32 inputs (P = 31, r = 5) are lowered
    to the word kernel, whose consumers read no staged tiles; the other
    operations and types of that size keep the staged word consumer.  At
    P = 24 (24 inputs) none of them does."""
    n = (1 << 20) + 37
    s = ar.Schedule(31, n, dtype, op, "generalized", jit="on", r=5)
    if s.dag_kernel_bytes() == 0:
        pytest.skip("NVRTC is not available on this host")
    low = s.lowering()
    assert low["tiling_ok"] == 1
    assert (low["word_sets"] > 0) == word and (low["dag_words"] == 0) == word, low
    small = ar.Schedule(24, n, dtype, op, "generalized", jit="on", r=4).lowering()
    assert small["word_sets"] == 0 and small["dag_words"] > 0


@pytest.mark.parametrize("P", [17, 18, 19, 24, 31])
def test_word_consumer_tiles_are_at_most_2_kib(lib, P):
    """Compiled programs of 17 to 32 inputs on the staged kernel take 2 KB
    tiles with as many stages as fit in the shared memory (at least 3, at
    most 8): at P = 17 six stages, not three of 4 KB."""
    low = ar.Schedule(P, (1 << 22) + 5, "float32", "sum", "generalized", jit="on", r=2).lowering()
    if low["dag_words"] == 0:
        pytest.skip("NVRTC is not available on this host")
    budget = 227 * 1024
    assert low["staged_tile_bytes"] == 2048
    assert low["staged_stages"] == min(8, (budget - 512) // (2048 * P)) >= 3


@pytest.mark.parametrize("algo,kw", [("ring", {}), ("rh", {}), ("rh", {"P": 7}), ("generalized", {}),
                                     ("generalized", {"group": "xor"})])
def test_fused_all_gathers_lower_to_the_copy_kernel(lib, algo, kw):
    """A fused all-gather's programs each copy one owner's chunk: one launch
    set on the copy kernel, whole 16-byte items that tile every chunk; the
    step form's rounds, the allreduce and the reduce-scatter keep their
    kernels."""
    kw = dict(kw)
    P = kw.pop("P", 8)
    n = (1 << 22) + 3
    low = ar.Schedule(P, n, "float32", "sum", algo, phase="all_gather", **kw).lowering()
    assert low["copy_sets"] == 1 and low["launch_sets"] == 1 and low["tiling_ok"] == 1
    for other in ({"phase": "all_gather", "form": "step"}, {"phase": "reduce_scatter"}, {}):
        assert ar.Schedule(P, n, "float32", "sum", algo, **other, **kw).lowering()["copy_sets"] == 0


@pytest.mark.parametrize("P,algo,kw,few", [(2, "ring", {}, 1), (3, "ring", {}, 1), (8, "ring", {}, 1), (16, "ring", {}, 1),
                                           (17, "ring", {}, 1), (64, "ring", {}, 1), (2, "rd", {}, 1),
                                           (8, "pipeline", {"blocks": 4}, 1),
                                           (2, "ring", {"form": "step"}, 0), (4, "ring", {"order": "fp32acc"}, 1),
                                           (16, "ring", {"order": "fp32acc"}, 1), (64, "ring", {"order": "fp32acc"}, 1),
                                           (4, "binomial", {}, 1), (8, "rh", {}, 1), (16, "rh", {}, 0),
                                           (8, "rh", {"form": "step"}, 0)])
def test_short_fused_chains_lower_to_the_few_input_kernel(lib, P, algo, kw, few):
    """Fused passes whose programs are all chains or fp32 accumulations (of
    up to 16 inputs at once, more in groups), or single trees (with chains)
    of up to 8, and too large for the chain word kernel, take the few-input
    kernel; larger trees and the step form's rounds keep theirs.  The items
    tile every range."""
    low = ar.Schedule(P, (1 << 24) + 3, "float32", "sum", algo, **kw).lowering()
    assert low["few_sets"] == few and low["tiling_ok"] == 1


def test_lowering_null_checks(lib):
    assert lib.ar_schedule_lowering(None, None) == 1
