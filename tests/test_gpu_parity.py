"""GPU parity: the engine's CUDA path against the CPU oracle, element by
element, through the C ABI.  Order-faithful results must be bit-identical to
the oracle's literal simulation (every dtype, every schedule); fp32-
accumulated results must stay within the normwise relative error the engine
promises (1e-6 fp32, 4e-3 bf16) of a float64 direct reduction."""

import numpy as np
import pytest

import ar_synth
import oracle
from oracle.chunking import ceil_log2
from oracle.direct import direct_f64, direct_int, normwise_rel_err
from oracle.elementops import Arith

from gpu_util import RankBufs, assert_bit_equal, engine, ensure_built, to_dev, to_host

pytestmark = pytest.mark.gpu

FORMS = ["fused", "step"]


@pytest.fixture(scope="module", autouse=True)
def built():
    ensure_built()
    import torch
    assert torch.cuda.is_available()


def check_faithful(bufs, dtype, op, algo, form, **kw):
    want = oracle.run(algo, bufs, Arith(op, dtype), **kw).bufs
    got = engine(bufs, dtype, op, algo, form=form, **kw)
    for r in range(len(bufs)):
        assert_bit_equal(got[r], want[r], dtype, f"{algo} {op} {dtype} {form} {kw} rank {r}")
    return got


# ---- configuration 1: ring, P = 3, 1024 int32 -------------------------------------------

@pytest.mark.parametrize("form", FORMS)
def test_config1_ring_int32(form):
    bufs = ar_synth.rank_inputs(3, 1024, "int32", "uniform_int")
    got = check_faithful(bufs, "int32", "sum", "ring", form)
    want = direct_int(bufs, "sum")
    for g in got:
        assert np.array_equal(g, want)


# ---- configuration 2: RH, RD, hybrid, binomial, P = 8, 2^20 fp32 -------------------------

CONFIG2 = [("rh", {}), ("rd", {}), ("binomial", {})] + [("hybrid", {"k1": k}) for k in range(4)]


@pytest.fixture(scope="module")
def config2_inputs():
    return ar_synth.rank_inputs(8, 1 << 20, "float32", "normal", sigma=1.0)


@pytest.mark.parametrize("form", FORMS)
@pytest.mark.parametrize("op", ["sum", "max"])
@pytest.mark.parametrize("algo,kw", CONFIG2)
def test_config2_power_of_two_schedules(config2_inputs, algo, kw, op, form):
    check_faithful(config2_inputs, "float32", op, algo, form, **kw)


@pytest.mark.parametrize("form", FORMS)
@pytest.mark.parametrize("P", [3, 6, 12, 13])
def test_non_power_of_two_folded_schedules(P, form):
    """RD, RH and the hybrid on any P through the preparation / finalization
    rounds around the largest power of two."""
    bufs = ar_synth.rank_inputs(P, 40003, "float32", "normal", sigma=1.0, seed=P)
    for algo, kw in (("rd", {}), ("rh", {}), ("hybrid", {"k1": 1})):
        for op in ("sum", "max"):
            check_faithful(bufs, "float32", op, algo, form, **kw)


@pytest.mark.parametrize("form", FORMS)
@pytest.mark.parametrize("P,m", [(2, 1), (5, 4), (8, 16), (13, 7)])
def test_pipelined_chain(P, m, form):
    bufs = ar_synth.rank_inputs(P, 100003, "bfloat16", "normal", sigma=1e-2, seed=m)
    for op in ("sum", "min"):
        check_faithful(bufs, "bfloat16", op, "pipeline", form, blocks=m)


# ---- configuration 3: generalized, P = 7 and 12 ----------------------------------------

@pytest.mark.parametrize("form", FORMS)
@pytest.mark.parametrize("n", [106, 1 << 20])
@pytest.mark.parametrize("P", [7, 12])
def test_config3_generalized_every_step_count(P, n, form):
    bufs = ar_synth.rank_inputs(P, n, "float32", "normal", sigma=1e-2)
    L = ceil_log2(P)
    for r in range(L + 1):
        check_faithful(bufs, "float32", "sum", "generalized", form, group="cyclic", r=r)


def test_config3_xor_group_rejected_for_p12():
    import collective_reduction_gb300 as ar
    with pytest.raises(ar.ArError) as e:
        ar.Plan(12, 106, "float32", "sum", "generalized", group="xor")
    assert e.value.name == "AR_ERR_UNSUPPORTED"


# ---- configuration 4: AHC, groups {2, 3}, 2^24 bf16 -------------------------------------

@pytest.fixture(scope="module")
def config4_inputs():
    return ar_synth.rank_inputs(5, 1 << 24, "bfloat16", "normal", sigma=1e-3)


@pytest.mark.parametrize("form", FORMS)
def test_config4_ahc_bf16(config4_inputs, form):
    check_faithful(config4_inputs, "bfloat16", "sum", "ahc", form, group_sizes=[2, 3])


def test_config4_ahc_fp32acc_within_tolerance(config4_inputs):
    got = engine(config4_inputs, "bfloat16", "sum", "ahc", group_sizes=[2, 3], order="fp32acc")
    ref = direct_f64(config4_inputs, "sum", "bfloat16")
    from oracle.elementops import bf16_to_f32
    for g in got:
        assert normwise_rel_err(bf16_to_f32(g), ref) <= 4e-3


# ---- configuration 5 (small points, full check) -----------------------------------------

@pytest.mark.parametrize("dtype", ["float32", "bfloat16"])
@pytest.mark.parametrize("P", [2, 8, 16, 64])
@pytest.mark.parametrize("nbytes", [1024, 65536, 1 << 20])
def test_config5_ring_small_sizes(P, nbytes, dtype):
    n = nbytes // (4 if dtype == "float32" else 2)
    bufs = ar_synth.rank_inputs(P, n, dtype, "normal", sigma=1e-3, seed=P)
    check_faithful(bufs, dtype, "sum", "ring", "fused")
    if nbytes <= 65536:
        check_faithful(bufs, dtype, "sum", "ring", "step")
    got = engine(bufs, dtype, "sum", "ring", order="fp32acc")
    ref = direct_f64(bufs, "sum", dtype)
    tol = 1e-6 if dtype == "float32" else 4e-3
    from oracle.elementops import bf16_to_f32
    for g in got:
        y = bf16_to_f32(g) if dtype == "bfloat16" else g
        assert normwise_rel_err(y, ref) <= tol


@pytest.mark.parametrize("dtype", ["float32", "bfloat16"])
@pytest.mark.parametrize("P", [2, 3, 7])
def test_many_items_per_cta(P, dtype):
    """Tens of rank-streaming items per CTA at small P, where consumer warps
    can drift a whole item apart: the pipeline's barriers must keep every
    item's result intact (full oracle comparison, plus the status word)."""
    n = (1 << 23) + 5
    bufs = ar_synth.rank_inputs(P, n, dtype, "normal", sigma=1e-2, seed=P + 100)
    check_faithful(bufs, dtype, "sum", "ring", "fused")
    got = engine(bufs, dtype, "sum", "ring", order="fp32acc")
    ref = direct_f64(bufs, "sum", dtype)
    from oracle.elementops import bf16_to_f32
    tol = 1e-6 if dtype == "float32" else 4e-3
    for g in got:
        assert normwise_rel_err(bf16_to_f32(g) if dtype == "bfloat16" else g, ref) <= tol


@pytest.mark.parametrize("dtype", ["float32", "bfloat16"])
@pytest.mark.parametrize("P,n,algo,form,kw", [
    (64, (1 << 20) + 7, "rh", "fused", {}),            # deep trees, 24 KB tiles, 1.1 waves of items
    (16, (3 << 20) + 3, "rh", "step", {}),             # 2.5 waves per round
    (5, (1 << 22) + 1, "ahc", "fused", {"group_sizes": [2, 3]}),
    (12, 2_000_003, "generalized", "step", {"r": 2}),  # versioned cyclic rounds
])
def test_partial_last_wave(P, n, algo, form, kw, dtype):
    """Sizes whose rank-streaming items end in a partial wave over the 152
    SMs (some CTAs take one item more than others), deep trees on 24 KB tiles
    and versioned rounds among them: full oracle comparison."""
    bufs = ar_synth.rank_inputs(P, n, dtype, "normal", sigma=1e-2, seed=P + 7)
    check_faithful(bufs, dtype, "sum", algo, form, **kw)


@pytest.mark.parametrize("dtype,form", [("float32", "fused"), ("bfloat16", "fused"), ("float32", "step")])
def test_bench_workload_at_full_size_sampled(dtype, form):
    """The bench's own workload and launch configuration — the ring over
    P = 8 x 256 MiB per rank, inputs drawn on the device as the bench draws
    them — checked on 4096 sampled elements of each of the 8 chunks of every
    rank: the sample keeps the chunk structure (a ceil split puts each
    chunk's elements in the same chunk), so the oracle's literal run on it
    owes exactly the sampled outputs, bit for bit."""
    import torch
    import bench
    import collective_reduction_gb300 as ar
    P = 8
    n = (256 << 20) // (2 if dtype == "bfloat16" else 4)
    src = ar_synth.device_inputs(P, n, dtype, sigma=1e-3, seed=0)
    sample_in, idx = bench.gather_sample(src, P, n, 4096, P)
    rb = RankBufs(P, n, dtype)
    for v, t in zip(rb.views, src):
        v.copy_(t)
    del src
    plan = ar.Plan(P, n, dtype, "sum", "ring", form=form)
    plan.execute(rb.views)
    plan.check()
    rb.check_guards("bench workload")
    want = oracle.run("ring", sample_in, Arith("sum", dtype)).bufs
    for r in range(P):
        got = to_host(rb.views[r].index_select(0, idx), dtype)
        assert_bit_equal(got, want[r], dtype, f"rank {r}")
    plan.close()
    del rb
    torch.cuda.empty_cache()


@pytest.mark.parametrize("algo,kw", [("ring", {}), ("ring", {"form": "step"}), ("rh", {}),
                                     ("generalized", {"r": 1, "op": "max", "jit": "on"})])
def test_rank_buffers_beyond_4_gib(algo, kw):
    """Rank buffers of 5 GiB + 12 bytes (byte offsets beyond 32 bits in every
    kernel's address arithmetic, a ragged tail): P = 2 (3 for the DAG plan),
    checked on 4096 sampled elements of every chunk, bit for bit the oracle."""
    import torch
    import bench
    import collective_reduction_gb300 as ar
    kw = dict(kw)
    op = kw.pop("op", "sum")
    P = 3 if algo == "generalized" else 2
    n = (5 << 30) // 4 + 3
    if torch.cuda.mem_get_info()[0] < P * n * 4 * 1.2:
        pytest.skip("not enough device memory")
    dev = ar_synth.device_inputs(P, n, "float32", sigma=1.0, seed=P)
    sample_in, idx = bench.gather_sample(dev, P, n, 4096, P)
    plan = ar.Plan(P, n, "float32", op, algo, **kw)
    plan.execute(dev)
    plan.check()
    want = oracle.run(algo, sample_in, Arith(op, "float32"),
                      **{k: v for k, v in kw.items() if k not in ("form", "jit")}).bufs
    for r in range(P):
        assert_bit_equal(to_host(dev[r].index_select(0, idx), "float32"), want[r], "float32", f"{algo} rank {r}")
    plan.close()
    del dev
    torch.cuda.empty_cache()


# ---- every (dtype, op) through a chain and a DAG program -------------------------------

@pytest.mark.parametrize("dtype", ["int32", "float32", "bfloat16"])
@pytest.mark.parametrize("op", ["sum", "prod", "max", "min"])
@pytest.mark.parametrize("algo,kw", [("ring", {}), ("rd", {}), ("generalized", {"r": 2}), ("binomial", {})])
def test_every_dtype_and_op(dtype, op, algo, kw):
    P = 4 if algo == "rd" else 5
    n = 4099
    dist = "small_int" if (dtype == "int32" and op == "prod") else ("uniform_int" if dtype == "int32" else "normal")
    bufs = ar_synth.rank_inputs(P, n, dtype, dist, sigma=1.5, seed=3)
    for form in FORMS:
        check_faithful(bufs, dtype, op, algo, form, **kw)


def test_special_values_bf16_and_fp32():
    """Ties, subnormals, infinities, NaN and signed zeros: P = 2 ring makes
    chunk 0 compute x1 (+) x0 and chunk 1 x0 (+) x1."""
    f32 = np.array([0.0, -0.0, 1e-40, -1e-40, 1.0, 1.0 + 2 ** -8, np.inf, -np.inf, np.nan, 3.4e38,
                    2 ** -126, 1.5, -2.5, 1e-45, 7.0, 0.1], dtype=np.float32)
    rng = np.random.default_rng(5)
    a = rng.permutation(np.concatenate([f32, -f32]))
    b = rng.permutation(np.concatenate([f32, f32[::-1]]))
    a = np.concatenate([a, b]).astype(np.float32)
    b = np.concatenate([b, a[:b.size]]).astype(np.float32)
    for op in ("sum", "prod", "max", "min"):
        check_faithful([a.copy(), b.copy()], "float32", op, "ring", "fused")
        from oracle.elementops import f32_to_bf16_rne
        check_faithful([f32_to_bf16_rne(a), f32_to_bf16_rne(b)], "bfloat16", op, "ring", "fused")


def test_bf16_rounding_edge_grid():
    """bf16 sums whose fp32 results sit exactly on, just above and just below
    bf16 rounding ties, including subnormal and overflow ranges."""
    rng = np.random.default_rng(9)
    hi = rng.integers(1, 0x7F7F, 4096, dtype=np.uint32).astype(np.uint16)
    lo = (hi.astype(np.uint32) - rng.integers(1, 24, 4096) * 0x80).clip(1, 0x7F7F).astype(np.uint16)
    sub = rng.integers(1, 0x80, 1024, dtype=np.uint32).astype(np.uint16)
    x = np.concatenate([hi, sub, hi | 0x8000]).astype(np.uint16)
    y = np.concatenate([lo, sub[::-1], lo]).astype(np.uint16)
    for op in ("sum", "prod"):
        check_faithful([x, y], "bfloat16", op, "ring", "fused")
        check_faithful([x, y], "bfloat16", op, "ring", "step")


@pytest.mark.parametrize("op", ["sum", "prod", "max", "min"])
@pytest.mark.parametrize("P,algo,kw", [(3, "ring", {}), (4, "rd", {}), (5, "generalized", {"r": 2}),
                                       (8, "rh", {}), (2, "ring", {})])
def test_bf16_every_bit_pattern_class(P, algo, kw, op):
    """Uniformly random 16-bit patterns (normal, subnormal, zero, infinite and
    NaN bf16 values of both signs) through the rank-streaming kernel's chains
    and trees and a DAG program, fused and step: bf16 sums and products are
    single bf16x2 instructions there, and must give the element op's bits
    (fp32 result rounded to bf16) everywhere; max / min take one bf16x2
    compare and must select as a > b ? a : b (a < b ? a : b) does."""
    n = 300_007
    rng = np.random.default_rng(1000 + P)
    bufs = [rng.integers(0, 1 << 16, n, dtype=np.uint32).astype(np.uint16) for _ in range(P)]
    for form in FORMS:
        check_faithful(bufs, "bfloat16", op, algo, form, **kw)


# ---- edge cases ---------------------------------------------------------------------------

@pytest.mark.parametrize("n", [0, 1, 3, 7, 1001, 4097])
@pytest.mark.parametrize("P", [1, 2, 7, 13])
def test_ragged_and_tiny_lengths(P, n):
    bufs = ar_synth.rank_inputs(P, n, "float32", "normal", sigma=1.0, seed=n)
    for form in FORMS:
        check_faithful(bufs, "float32", "sum", "ring", form)
        check_faithful(bufs, "float32", "sum", "generalized", form, r=min(1, ceil_log2(P)))


def test_unaligned_buffers_take_elementwise_path():
    """Buffers one element past a 16-byte boundary: the element-wise path,
    the skipped leading element checked with the guard band before it."""
    P, n = 6, 3001
    bufs = ar_synth.rank_inputs(P, n, "float32", "normal", seed=4)
    want = oracle.run("generalized", bufs, Arith("sum", "float32"), r=1).bufs
    for form in FORMS:
        got = engine(bufs, "float32", "sum", "generalized", offset=1, r=1, form=form)
        for r in range(P):
            assert_bit_equal(got[r], want[r], "float32", f"unaligned {form} rank {r}")


@pytest.mark.parametrize("dtype", ["float32", "int32"])
@pytest.mark.parametrize("P,algo,kw", [(3, "ring", {}), (8, "ring", {}), (20, "ring", {}),
                                       (8, "pipeline", {"blocks": 3}), (8, "ring", {"form": "step"})])
def test_unaligned_chains_of_4_byte_elements(P, algo, kw, dtype):
    """Buffers one element off a 16-byte boundary: a pass of chains over
    4-byte elements (every element on a 32-bit word) runs on the chain word
    kernel, every other pass element by element; bit for bit the oracle,
    the skipped leading element inside the guard band."""
    n = 100_003
    dist = "uniform_int" if dtype == "int32" else "normal"
    bufs = ar_synth.rank_inputs(P, n, dtype, dist, sigma=1.0, seed=P + 55)
    want = oracle.run(algo, bufs, Arith("sum", dtype), **{k: v for k, v in kw.items() if k != "form"}).bufs
    got = engine(bufs, dtype, "sum", algo, offset=1, **kw)
    for r in range(P):
        assert_bit_equal(got[r], want[r], dtype, f"unaligned {algo} {kw} rank {r}")


@pytest.mark.parametrize("dtype", ["bfloat16", "float32"])
@pytest.mark.parametrize("P,algo,kw", [(5, "ring", {}), (8, "ring", {}), (64, "ring", {}),
                                       (5, "ahc", {"group_sizes": [2, 3]}), (3, "ring", {}), (4, "ring", {})])
def test_fp32acc_same_bits_in_every_kernel(P, algo, kw, dtype):
    """The fp32-accumulate order is the engine's own and the same in every
    kernel: the few-input kernel (P = 3 ... 8) and the rank-streaming kernel
    (P = 64 at this size; bf16 on 24 KB tiles, fp32 on 32 KB) must give
    exactly the bits of the element-wise kernel, which unaligned buffers
    take.  test_fp32acc_grouped_on_the_few_input_kernel covers the grouped
    variant."""
    n = 300_007
    bufs = ar_synth.rank_inputs(P, n, dtype, "normal", sigma=1e-2, seed=P + 3)
    fast = engine(bufs, dtype, "sum", algo, order="fp32acc", **kw)
    slow = engine(bufs, dtype, "sum", algo, offset=1, order="fp32acc", **kw)  # not 16-byte aligned
    for r in range(P):
        assert_bit_equal(slow[r], fast[r], dtype, f"{algo} P={P} rank {r}")


@pytest.mark.parametrize("dtype", ["bfloat16", "float32"])
@pytest.mark.parametrize("order", ["fp32acc", "faithful"])
def test_fp32acc_grouped_on_the_few_input_kernel(order, dtype):
    """Chains and fp32 accumulations of 64 inputs in a set of at least 1.5
    GiB run on the few-input kernel's grouped variant (8 inputs' loads in
    flight at a time, folded in the program's order across the groups): bit
    for bit the element-wise kernel, which the same plan takes for buffers
    one element off the 16-byte grid (itself checked against the oracle in
    the other tests), every element of every rank, guard bands intact."""
    import torch
    import collective_reduction_gb300 as ar
    P, n = 64, ((3 << 21) + 64) * (2 if dtype == "bfloat16" else 1)  # 24 MiB per rank
    plan = ar.Plan(P, n, dtype, "sum", "ring", order=order)
    assert plan.info()["kernels"] & ar.KERNEL_FEW, plan.info()["kernels"]
    tdt = torch.bfloat16 if dtype == "bfloat16" else torch.float32
    itype = torch.int16 if dtype == "bfloat16" else torch.int32
    fast, slow = RankBufs(P, n, dtype), RankBufs(P, n, dtype, offset=1)
    gen = torch.Generator(device="cuda").manual_seed(64)
    for r in range(P):
        x = (torch.randn(n, device="cuda", generator=gen) * 1e-2).to(tdt)
        fast.views[r].copy_(x)
        slow.views[r].copy_(x)
    plan.execute(fast.views)
    plan.execute(slow.views)
    torch.cuda.synchronize()
    plan.check()
    plan.close()
    fast.check_guards("grouped")
    slow.check_guards("element-wise")
    for r in range(P):
        assert torch.equal(fast.views[r].view(itype), slow.views[r].view(itype)), f"{order} {dtype} rank {r}"


@pytest.mark.parametrize("form", FORMS)
def test_p64_latency_optimal_max(form):
    """P = 64, r = ceil(log2 P): a rank-specific tree per rank (max keeps the
    operand order, so no tree merges)."""
    P, n = 64, 640
    bufs = ar_synth.rank_inputs(P, n, "float32", "normal", seed=64)
    check_faithful(bufs, "float32", "max", "generalized", form, r=6)
    check_faithful(bufs, "float32", "sum", "generalized", form, r=6, group="xor")


def test_invalid_buffers_rejected():
    import torch
    import collective_reduction_gb300 as ar
    t = [torch.zeros(100, device="cuda") for _ in range(3)]
    plan = ar.Plan(3, 100, "float32", "sum", "ring")
    for bad in ([t[0], t[0], t[1]], [t[0], t[1], t[0][10:]]):
        with pytest.raises(ar.ArError) as e:
            plan.execute(bad)
        assert e.value.name == "AR_ERR_INVALID_ARG"
    with pytest.raises(ar.ArError):
        plan.execute([t[0], t[1], 0])
    plan.close()


def _segment_of(t):
    """(address, size) of the caching allocator's segment holding tensor t."""
    import torch
    p = t.data_ptr()
    for seg in torch.cuda.memory_snapshot():
        if seg["address"] <= p < seg["address"] + seg["total_size"]:
            return seg["address"], seg["total_size"]
    return None


def test_buffer_residency_checked_before_any_launch():
    """ar_plan_check_buffers applies ar_execute's buffer checks and launches
    nothing: device memory of the plan's device passes; pageable host memory,
    pinned host memory and a buffer whose n elements run past the allocation
    holding it are refused.  (Tested through the check alone, so that no bad
    pointer could reach a kernel even if the check regressed.)"""
    import os

    import torch
    import collective_reduction_gb300 as ar
    P, n = 3, 1 << 20
    plan = ar.Plan(P, n, "float32", "sum", "ring")
    good = [torch.zeros(n, device="cuda") for _ in range(P)]
    assert plan.check_buffers(good) == "AR_OK"
    pageable = np.zeros(n, np.float32)
    assert plan.check_buffers([good[0], good[1], pageable.ctypes.data]) == "AR_ERR_INVALID_ARG"
    pinned = torch.zeros(n).pin_memory()
    assert plan.check_buffers([good[0], pinned.data_ptr(), good[2]]) == "AR_ERR_INVALID_ARG"
    assert plan.check_buffers([good[0], good[1], 0]) == "AR_ERR_INVALID_ARG"
    assert plan.check_buffers([good[0], good[1], good[1].data_ptr() + 4096]) == "AR_ERR_INVALID_ARG"  # overlap
    if "expandable_segments:True" not in os.environ.get("PYTORCH_CUDA_ALLOC_CONF", ""):
        big = torch.empty(24 << 20, dtype=torch.uint8, device="cuda")
        seg = _segment_of(big)
        assert seg is not None
        base, size = seg
        inside = base + size - 4 * n            # the last n elements of the segment: fine
        past = inside + 4096                    # starts inside, ends 4 KiB past the segment
        assert plan.check_buffers([good[0], good[1], inside]) == "AR_OK"
        assert plan.check_buffers([good[0], good[1], past]) == "AR_ERR_INVALID_ARG"
    plan.close()


def test_execute_host_end_to_end():
    import torch
    import collective_reduction_gb300 as ar
    P, n = 8, 1 << 16
    bufs = ar_synth.rank_inputs(P, n, "float32", "normal", seed=8)
    want = oracle.run("ring", bufs, Arith("sum", "float32")).bufs
    host = [torch.from_numpy(b.copy()).pin_memory() for b in bufs]
    rb = RankBufs(P, n, "float32")
    dev = rb.views
    plan = ar.Plan(P, n, "float32", "sum", "ring")
    plan.execute_host(host, dev)
    plan.check()
    rb.check_guards("e2e")
    for r in range(P):
        assert_bit_equal(host[r].numpy(), want[r], "float32", f"e2e rank {r}")
        assert_bit_equal(dev[r].cpu().numpy(), want[r], "float32", f"e2e dev rank {r}")
    plan.close()


@pytest.mark.parametrize("order", ["faithful", "fp32acc"])
def test_execute_host_pipelined_windows(order):
    """Large enough for the windowed host path (copies overlapped with the
    reduction, several windows), ragged so windows also carry edge items."""
    import torch
    import collective_reduction_gb300 as ar
    P, n = 7, 10_000_003
    bufs = ar_synth.rank_inputs(P, n, "float32", "normal", sigma=1e-2, seed=77)
    host = [torch.from_numpy(b.copy()).pin_memory() for b in bufs]
    rb = RankBufs(P, n, "float32")
    dev = rb.views
    plan = ar.Plan(P, n, "float32", "sum", "ring", order=order)
    for _ in range(2):  # second call reuses the plan's streams and events
        for r in range(P):
            host[r].copy_(torch.from_numpy(bufs[r]))
        plan.execute_host(host, dev)
        plan.check()
        rb.check_guards("windows")
        if order == "faithful":
            want = oracle.run("ring", bufs, Arith("sum", "float32")).bufs
            for r in range(P):
                assert_bit_equal(host[r].numpy(), want[r], "float32", f"host rank {r}")
                assert_bit_equal(dev[r].cpu().numpy(), want[r], "float32", f"dev rank {r}")
        else:
            ref = direct_f64(bufs, "sum", "float32")
            for r in range(P):
                assert normwise_rel_err(host[r].numpy(), ref) <= 1e-6
                assert np.array_equal(host[r].numpy(), dev[r].cpu().numpy())
    plan.close()


@pytest.mark.parametrize("P,n,dtype,algo", [(64, 1 << 20, "float32", "rh"), (8, (1 << 24) + 3, "bfloat16", "ring")])
def test_execute_host_windows_trees_and_bf16(P, n, dtype, algo):
    """Windowed host path for a deep-tree plan (24 KB tiles) and a ragged
    bf16 ring: every window's copies hold its items, so the results match
    the oracle bit for bit."""
    import torch
    import collective_reduction_gb300 as ar
    assert ar.Schedule(P, n, dtype, "sum", algo).lowering()["windows"] >= 2
    bufs = ar_synth.rank_inputs(P, n, dtype, "normal", sigma=1e-2, seed=P + 31)
    tdt = torch.bfloat16 if dtype == "bfloat16" else torch.float32
    host = [torch.from_numpy(np.ascontiguousarray(b).view(np.int16).copy()).view(tdt).pin_memory()
            if dtype == "bfloat16" else torch.from_numpy(b.copy()).pin_memory() for b in bufs]
    rb = RankBufs(P, n, dtype)
    dev = rb.views
    plan = ar.Plan(P, n, dtype, "sum", algo)
    plan.execute_host(host, dev)
    plan.check()
    rb.check_guards("windows")
    want = oracle.run(algo, bufs, Arith("sum", dtype)).bufs
    for r in range(P):
        got = host[r].view(torch.int16).numpy().view(np.uint16) if dtype == "bfloat16" else host[r].numpy()
        assert_bit_equal(got, want[r], dtype, f"host rank {r}")
    plan.close()


@pytest.mark.parametrize("algo,phase", [("ring", "reduce_scatter"), ("ring", "all_gather"),
                                         ("rh", "reduce_scatter")])
def test_execute_host_windows_for_the_halves(algo, phase):
    """The windowed host path for one half of the allreduce: a fused
    reduce-scatter writes only the owners' chunks (the rest come back as they
    went in), an all-gather every non-owner's."""
    import torch
    import collective_reduction_gb300 as ar
    P, n = 8, (1 << 23) + 5
    assert ar.Schedule(P, n, "float32", "sum", algo, phase=phase).lowering()["windows"] >= 2
    bufs = ar_synth.rank_inputs(P, n, "float32", "normal", sigma=1e-2, seed=17)
    host = [torch.from_numpy(b.copy()).pin_memory() for b in bufs]
    rb = RankBufs(P, n, "float32")
    dev = rb.views
    plan = ar.Plan(P, n, "float32", "sum", algo, phase=phase)
    plan.execute_host(host, dev)
    plan.check()
    rb.check_guards("windows")
    want = oracle.run(algo, bufs, Arith("sum", "float32"), phase=phase)
    if phase == "reduce_scatter":
        for r, lo, hi in want.info["owner"]:
            assert_bit_equal(host[r].numpy()[lo:hi], want.bufs[r][lo:hi], "float32", f"owner {r}")
    else:
        for r in range(P):
            assert_bit_equal(host[r].numpy(), want.bufs[r], "float32", f"host rank {r}")
    plan.close()


def test_repeated_execute_and_streams():
    """Back-to-back executes on a side stream, then on the default stream."""
    import torch
    import collective_reduction_gb300 as ar
    P, n = 8, 1 << 18
    bufs = ar_synth.rank_inputs(P, n, "int32", "small_int", seed=2)
    plan = ar.Plan(P, n, "int32", "sum", "ring")
    rb = RankBufs.from_host(bufs, "int32")
    dev = rb.views
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(3):
            plan.execute(dev)
    torch.cuda.current_stream().wait_stream(s)
    plan.execute(dev)
    torch.cuda.synchronize()
    plan.check()
    # four allreduces: each multiplies the sum by P
    x = direct_int(bufs, "sum").astype(np.int64)
    for _ in range(3):
        x = (x * P)
    want = (x.astype(np.int64) & 0xFFFFFFFF).astype(np.uint32).view(np.int32)
    rb.check_guards("repeated")
    for t in dev:
        assert np.array_equal(to_host(t, "int32"), want)
    plan.close()


# ---- reduce-scatter / all-gather halves -------------------------------------------------

SPLIT = [("ring", {}), ("rh", {}), ("generalized", {"group": "cyclic"})]


def _owners(algo, P, n, kw):
    """(rank, lo, hi): who holds [lo, hi) after the oracle's reduce-scatter."""
    zeros = [np.zeros(n, np.int32)] * P
    return oracle.run(algo, zeros, Arith("sum", "int32"), phase="reduce_scatter", **kw).info["owner"]


@pytest.mark.parametrize("form", FORMS)
@pytest.mark.parametrize("dtype", ["int32", "float32", "bfloat16"])
@pytest.mark.parametrize("P", [3, 8, 12])
def test_reduce_scatter_owned_chunks(P, dtype, form):
    """Each owner's chunk bit-identical to the oracle's reduce-scatter; the
    other chunks are unspecified and not compared."""
    n = 100003
    dist = "uniform_int" if dtype == "int32" else "normal"
    bufs = ar_synth.rank_inputs(P, n, dtype, dist, sigma=1e-2, seed=P + 7)
    cases = SPLIT + ([("generalized", {"group": "xor"})] if P & (P - 1) == 0 else [])
    for algo, kw in cases:
        for op in ("sum", "max"):
            res = oracle.run(algo, bufs, Arith(op, dtype), phase="reduce_scatter", **kw)
            got = engine(bufs, dtype, op, algo, form=form, phase="reduce_scatter", **kw)
            for rank, lo, hi in res.info["owner"]:
                assert_bit_equal(got[rank][lo:hi], res.bufs[rank][lo:hi], dtype,
                                 f"{algo} {kw} {op} rank {rank} [{lo}, {hi})")


@pytest.mark.parametrize("dtype", ["float32", "bfloat16"])
def test_reduce_scatter_fp32acc_within_tolerance(dtype):
    P, n = 8, (1 << 22) + 9
    bufs = ar_synth.rank_inputs(P, n, dtype, "normal", sigma=1e-2, seed=41)
    ref = direct_f64(bufs, "sum", dtype)
    tol = 1e-6 if dtype == "float32" else 4e-3
    from oracle.elementops import bf16_to_f32
    for algo, kw in SPLIT:
        owner = _owners(algo, P, n, kw)
        got = engine(bufs, dtype, "sum", algo, order="fp32acc", phase="reduce_scatter", **kw)
        y = np.empty(n, np.float64)
        for rank, lo, hi in owner:
            g = got[rank][lo:hi]
            y[lo:hi] = bf16_to_f32(g) if dtype == "bfloat16" else g
        assert normwise_rel_err(y, ref) <= tol, algo


@pytest.mark.parametrize("form", FORMS)
@pytest.mark.parametrize("dtype", ["int32", "float32", "bfloat16"])
@pytest.mark.parametrize("P", [2, 7, 12, 16])
def test_all_gather_spreads_owned_chunks(P, dtype, form):
    """Every rank ends with the owners' chunks, bit for bit; what the other
    chunks held beforehand (here a sentinel) must not survive anywhere."""
    n = 77777
    dist = "uniform_int" if dtype == "int32" else "normal"
    src = ar_synth.rank_inputs(P, n, dtype, dist, sigma=1.0, seed=P + 9)
    cases = SPLIT + ([("generalized", {"group": "xor"})] if P & (P - 1) == 0 else [])
    for algo, kw in cases:
        owner = _owners(algo, P, n, kw)
        bufs = [np.full_like(b, 0x7BCD if dtype == "bfloat16" else -12345) for b in src]
        for rank, lo, hi in owner:
            bufs[rank][lo:hi] = src[rank][lo:hi]
        want = oracle.run(algo, bufs, Arith("sum", dtype), phase="all_gather", **kw).bufs
        got = engine(bufs, dtype, "sum", algo, form=form, phase="all_gather", **kw)
        for r in range(P):
            assert_bit_equal(got[r], want[r], dtype, f"{algo} {kw} rank {r}")


@pytest.mark.parametrize("P,algo,kw,dtype,offset", [(64, "ring", {}, "float32", 0), (33, "rh", {}, "bfloat16", 0),
                                                     (8, "generalized", {"group": "xor"}, "float32", 0),
                                                     (8, "ring", {}, "bfloat16", 1), (3, "ring", {}, "int32", 0)])
def test_fused_all_gathers_run_on_the_copy_kernel(P, algo, kw, dtype, offset):
    """Fused all-gathers run on the copy kernel (one input chunk stored to
    every other rank, 2048 threads per SM): bit for bit the oracle's result
    at a length of several 32 KB items with a ragged tail, 63 outputs per
    item at P = 64, guard bands intact; with buffers one element off the
    16-byte grid the plan takes the element-wise fallback instead."""
    import collective_reduction_gb300 as ar
    n = (3 << 16) + 7 if P <= 8 else (1 << 14) + 3
    dist = "uniform_int" if dtype == "int32" else "normal"
    src = ar_synth.rank_inputs(P, n, dtype, dist, sigma=1.0, seed=P + 41)
    plan = ar.Plan(P, n, dtype, "sum", algo, phase="all_gather", **kw)
    assert plan.info()["kernels"] & ar.KERNEL_COPY, plan.info()["kernels"]
    plan.close()
    want = oracle.run(algo, src, Arith("sum", dtype), phase="all_gather", **kw).bufs
    got = engine(src, dtype, "sum", algo, offset=offset, phase="all_gather", **kw)
    for r in range(P):
        assert_bit_equal(got[r], want[r], dtype, f"{algo} {kw} rank {r}")


@pytest.mark.parametrize("P,algo,op,dtype,offset", [(2, "ring", "sum", "float32", 0), (3, "ring", "max", "bfloat16", 0),
                                                     (4, "ring", "avg", "float32", 0), (4, "ring", "prod", "int32", 0),
                                                     (2, "rd", "sum", "bfloat16", 0), (3, "pipeline", "min", "float32", 0),
                                                     (4, "ring", "sum", "bfloat16", 1), (4, "ring", "avg", "bfloat16", 0),
                                                     (8, "rh", "sum", "float32", 0), (8, "binomial", "max", "bfloat16", 0),
                                                     (7, "rh", "avg", "float32", 0), (8, "rd", "prod", "int32", 0),
                                                     (6, "ahc", "sum", "bfloat16", 0), (5, "generalized", "min", "float32", 0),
                                                     (8, "hybrid", "sum", "bfloat16", 1)])
def test_short_chains_run_on_the_few_input_kernel(P, algo, op, dtype, offset):
    """Fused passes of chains of up to 16 inputs and single trees of up to 8
    leaves run on the few-input kernel (a CTA per 16 KB item, every input's
    vectors loaded before the fold; a tree's stack in registers): bit for
    bit the oracle's chains and trees, avg divided where they complete,
    over several items and a ragged tail, guard bands intact; one element off
    the 16-byte grid the plan takes the element-wise fallback instead."""
    import collective_reduction_gb300 as ar
    n = (5 << 15) + 11
    kw = {"pipeline": {"blocks": 3}, "ahc": {"group_sizes": [2, 4]}, "hybrid": {"k1": 1}}.get(algo, {})
    dist = "uniform_int" if dtype == "int32" else "normal"
    bufs = ar_synth.rank_inputs(P, n, dtype, dist, sigma=1.0, seed=P + 77)
    plan = ar.Plan(P, n, dtype, op, algo, **kw)
    assert plan.info()["kernels"] & ar.KERNEL_FEW, plan.info()["kernels"]
    plan.close()
    want = oracle.run(algo, bufs, Arith(op, dtype), **kw).bufs
    got = engine(bufs, dtype, op, algo, offset=offset, **kw)
    for r in range(P):
        assert_bit_equal(got[r], want[r], dtype, f"{algo} {op} rank {r}")


# ---- avg: the sum divided by P where it completes ---------------------------------------

AVG_CASES = [("ring", {}), ("binomial", {}), ("rd", {}), ("rh", {}), ("hybrid", {"k1": 1}),
             ("generalized", {"r": 0}), ("generalized", {"r": 2}), ("ahc", {"group_sizes": [2, 3, 2]}),
             ("pipeline", {"blocks": 3})]


@pytest.mark.parametrize("form", FORMS)
@pytest.mark.parametrize("dtype", ["float32", "bfloat16"])
def test_avg_every_schedule(dtype, form):
    P = 7
    for n in (5, 30011):
        bufs = ar_synth.rank_inputs(P, n, dtype, "normal", sigma=1.0, seed=n)
        for algo, kw in AVG_CASES:
            check_faithful(bufs, dtype, "avg", algo, form, **kw)


@pytest.mark.parametrize("dtype", ["float32", "bfloat16"])
def test_avg_fp32acc_and_halves(dtype):
    P, n = 8, (1 << 20) + 3
    bufs = ar_synth.rank_inputs(P, n, dtype, "normal", sigma=1e-2, seed=5)
    ref = direct_f64(bufs, "avg", dtype)
    tol = 1e-6 if dtype == "float32" else 4e-3
    from oracle.elementops import bf16_to_f32
    got = engine(bufs, dtype, "avg", "ring", order="fp32acc")
    for g in got:
        assert normwise_rel_err(bf16_to_f32(g) if dtype == "bfloat16" else g, ref) <= tol
    for form in FORMS:
        for algo, kw in SPLIT:
            res = oracle.run(algo, bufs, Arith("avg", dtype), phase="reduce_scatter", **kw)
            got = engine(bufs, dtype, "avg", algo, form=form, phase="reduce_scatter", **kw)
            for rank, lo, hi in res.info["owner"]:
                assert_bit_equal(got[rank][lo:hi], res.bufs[rank][lo:hi], dtype, f"{algo} {form} rank {rank}")


@pytest.mark.parametrize("dtype", ["float32", "bfloat16"])
@pytest.mark.parametrize("P,algo,form", [(2, "ring", "fused"), (4, "ring", "fused"), (8, "ring", "fused"),
                                         (8, "rh", "step"), (16, "binomial", "fused"), (3, "ring", "fused")])
def test_avg_special_values_and_subnormal_quotients(P, algo, form, dtype):
    """avg over random bit patterns (normal, subnormal, zero, infinite and NaN
    values of both signs) and over tiny sums whose quotient is subnormal and
    sits on or beside a rounding tie: at P = 2^k the kernels multiply by the
    exact reciprocal, which must give the IEEE quotient's bits everywhere; at
    P = 3 they divide."""
    n = 200_003
    rng = np.random.default_rng(31 * P + len(dtype))
    if dtype == "float32":
        rand = [rng.integers(0, 1 << 32, n, dtype=np.uint64).astype(np.uint32).view(np.float32) for _ in range(P)]
        tiny = [(rng.integers(-64, 64, n) * np.float32(2.0 ** -149)).astype(np.float32) for _ in range(P)]
    else:
        rand = [rng.integers(0, 1 << 16, n, dtype=np.uint32).astype(np.uint16) for _ in range(P)]
        tiny = [(rng.integers(0, 64, n, dtype=np.uint32) | (rng.integers(0, 2, n, dtype=np.uint32) << 15))
                .astype(np.uint16) for _ in range(P)]
    for bufs in (rand, tiny):
        check_faithful([b.copy() for b in bufs], dtype, "avg", algo, form)


def test_avg_unaligned_and_int32_refused():
    import collective_reduction_gb300 as ar
    P, n = 3, 1001
    bufs = ar_synth.rank_inputs(P, n, "float32", "normal", sigma=1.0, seed=8)
    want = oracle.run("ring", bufs, Arith("avg", "float32")).bufs
    got = engine(bufs, "float32", "avg", "ring", offset=1)  # 4-byte offset: element-wise path
    for r in range(P):
        assert_bit_equal(got[r], want[r], "float32", f"rank {r}")
    with pytest.raises(ar.ArError):
        ar.Plan(P, n, "int32", "avg", "ring")


def test_kernel_choice_per_program_kind():
    """Chains of up to 16 inputs and single trees of up to 8 leaves take a
    CTA per item (few-input kernel); larger single trees stream rank tiles
    (rank-streaming kernel); rank-specific DAGs stage an item's tiles
    (staged kernel); tiny or unaligned ranges go element by element."""
    import collective_reduction_gb300 as ar
    n = 1 << 20
    for algo, kw in (("ring", {}), ("rh", {}), ("binomial", {}), ("rd", {}), ("ahc", {"group_sizes": [4, 4]})):
        k = ar.Plan(8, n, "float32", "sum", algo, **kw).info()["kernels"]
        assert k == ar.KERNEL_FEW, (algo, k)
    for algo, kw in (("rh", {}), ("binomial", {}), ("ahc", {"group_sizes": [8, 8]})):
        k = ar.Plan(16, n, "float32", "sum", algo, **kw).info()["kernels"]
        assert k == ar.KERNEL_STREAM, (algo, k)
    # 30 chunks of 2^20 elements: unaligned chunk edges go element-wise
    k = ar.Plan(8, n, "float32", "sum", "ahc", group_sizes=[3, 5]).info()["kernels"]
    assert k == ar.KERNEL_FEW | ar.KERNEL_ELEMENTWISE, k
    assert ar.Plan(8, n, "bfloat16", "sum", "rh").info()["kernels"] == ar.KERNEL_FEW
    assert ar.Plan(7, 7 * 4096, "float32", "max", "generalized", r=3).info()["kernels"] & ar.KERNEL_STAGED
    assert ar.Plan(3, 5, "float32", "sum", "ring").info()["kernels"] == ar.KERNEL_ELEMENTWISE


@pytest.mark.parametrize("dtype", ["float32", "bfloat16"])
@pytest.mark.parametrize("algo,kw", [("rh", {}), ("binomial", {}), ("generalized", {"r": 0}),
                                     ("ahc", {"group_sizes": [2, 6]}), ("rh", {"phase": "reduce_scatter"})])
def test_streamed_trees_many_items(algo, kw, dtype):
    """Single trees on the rank-streaming kernel over many items per CTA,
    with a ragged tail: bit-identical to the oracle on the owned / all
    elements.  For bf16 the whole tiles and each range's partial last tile
    run different compilations of the tree consumer (without and with the
    per-vector bounds test); this size gives every rank both."""
    P, n = 8, (1 << 22) + 77
    bufs = ar_synth.rank_inputs(P, n, dtype, "normal", sigma=1e-2, seed=17)
    res = oracle.run(algo, bufs, Arith("sum", dtype), **kw)
    got = engine(bufs, dtype, "sum", algo, **kw)
    if kw.get("phase") == "reduce_scatter":
        for r, lo, hi in res.info["owner"]:
            assert_bit_equal(got[r][lo:hi], res.bufs[r][lo:hi], dtype, f"{algo} rank {r}")
    else:
        for r in range(P):
            assert_bit_equal(got[r], res.bufs[r], dtype, f"{algo} {kw} rank {r}")


@pytest.mark.parametrize("P", [16, 32, 64])
@pytest.mark.parametrize("dtype,op", [("float32", "sum"), ("bfloat16", "sum"), ("int32", "max")])
def test_trees_with_the_stack_in_tensor_memory(P, dtype, op):
    """Single trees of more than 8 leaves keep their stack in tensor memory
    (the lowering reports it): RH, binomial, AHC over two groups and RH's
    reduce-scatter, several items per CTA with a ragged tail, bit for bit the
    oracle; guard bands and the status word clean."""
    import collective_reduction_gb300 as ar
    n = (1 << 21) + 13 if P < 64 else (1 << 20) + 13
    assert ar.Schedule(P, n, dtype, op, "rh").lowering()["stream_tmem"] == 1
    dist = "uniform_int" if dtype == "int32" else "normal"
    bufs = ar_synth.rank_inputs(P, n, dtype, dist, sigma=1e-2, seed=P + 303)
    for algo, kw in (("rh", {}), ("binomial", {}), ("ahc", {"group_sizes": [P // 2, P - P // 2]}),
                     ("rh", {"phase": "reduce_scatter"})):
        res = oracle.run(algo, bufs, Arith(op, dtype), **kw)
        got = engine(bufs, dtype, op, algo, **kw)
        if kw.get("phase") == "reduce_scatter":
            for r, lo, hi in res.info["owner"]:
                assert_bit_equal(got[r][lo:hi], res.bufs[r][lo:hi], dtype, f"{algo} {kw} rank {r}")
        else:
            for r in range(P):
                assert_bit_equal(got[r], res.bufs[r], dtype, f"{algo} {kw} rank {r}")


@pytest.mark.parametrize("P,n,dtype,op,algo,kw", [
    (16, 1 << 18, "float32", "avg", "ring", {}),              # 1 MiB per rank, the avg division
    (64, 4096 + 64, "bfloat16", "sum", "ring", {}),           # 8 KiB per rank, ragged chunk edges
    (16, 257 * 16, "int32", "prod", "ring", {}),
    (16, 1 << 16, "float32", "max", "pipeline", {"blocks": 5}),
    (12, (1 << 18) + 3, "bfloat16", "min", "ring", {}),
])
def test_chain_word_passes(P, n, dtype, op, algo, kw):
    """Small and mid-sized fused chain passes on the chain word kernel (the
    plan reports it): every op, bf16 pairs in one word, the avg division, a
    pipelined chain, ragged edges on the element-wise kernel; bit for bit the
    oracle."""
    import collective_reduction_gb300 as ar
    assert ar.Plan(P, n, dtype, op, algo, **kw).info()["kernels"] & ar.KERNEL_CHAIN_WORD
    dist = "small_int" if (dtype == "int32" and op == "prod") else ("uniform_int" if dtype == "int32" else "normal")
    bufs = ar_synth.rank_inputs(P, n, dtype, dist, sigma=1.0, seed=P + 404)
    check_faithful(bufs, dtype, op, algo, "fused", **kw)


# ---- run-time compiled DAG kernels --------------------------------------------------------

JIT_CASES = [("generalized", 7, "sum", {"r": 1}), ("generalized", 7, "sum", {"r": 3}), ("rd", 8, "max", {}),
             ("generalized", 12, "min", {"r": 2}), ("generalized", 7, "avg", {"r": 2}),
             ("hybrid", 8, "max", {"k1": 1}), ("generalized", 7, "max", {"r": 3, "form": "step"}),
             ("generalized", 12, "sum", {"r": 4, "form": "step"})]


@pytest.mark.parametrize("dtype", ["int32", "float32", "bfloat16"])
@pytest.mark.parametrize("algo,P,op,kw", JIT_CASES)
def test_dag_kernel_jit_bit_exact(algo, P, op, kw, dtype):
    """DAG programs as run-time compiled straight-line code give the
    interpreter's bits, which are the oracle's; the plan reports which path
    it took."""
    import torch

    import collective_reduction_gb300 as ar
    if op == "avg" and dtype == "int32":
        pytest.skip("avg has no integer form")
    n = 50021
    dist = "uniform_int" if dtype == "int32" else "normal"
    bufs = ar_synth.rank_inputs(P, n, dtype, dist, sigma=1.0, seed=P + len(kw))
    okw = {k: v for k, v in kw.items() if k != "form"}
    want = oracle.run(algo, bufs, Arith(op, dtype), **okw).bufs
    for jit in ("on", "off"):
        plan = ar.Plan(P, n, dtype, op, algo, jit=jit, **kw)
        info = plan.info()
        staged = bool(info["kernels"] & ar.KERNEL_STAGED)
        assert bool(info["kernels"] & ar.KERNEL_DAG_JIT) == (staged and jit == "on"), (jit, info["kernels"])
        rb = RankBufs.from_host(bufs, dtype)
        plan.execute(rb.views)
        torch.cuda.synchronize()
        plan.check()
        rb.check_guards(f"{algo} {kw} jit={jit}")
        for r in range(P):
            assert_bit_equal(to_host(rb.views[r], dtype), want[r], dtype, f"{algo} {kw} jit={jit} rank {r}")
        plan.close()


def test_dag_kernel_jit_auto_threshold():
    import collective_reduction_gb300 as ar
    small = ar.Plan(7, 7 * 1024, "float32", "sum", "generalized", r=3).info()["kernels"]
    large = ar.Plan(7, 1 << 22, "float32", "sum", "generalized", r=3).info()["kernels"]
    assert small & ar.KERNEL_STAGED and not small & ar.KERNEL_DAG_JIT
    assert large & ar.KERNEL_STAGED and large & ar.KERNEL_DAG_JIT
    off = ar.Plan(7, 1 << 22, "float32", "sum", "generalized", r=3, jit="off").info()["kernels"]
    assert off & ar.KERNEL_STAGED and not off & ar.KERNEL_DAG_JIT


WORD_CASES = [(31, "generalized", "sum", {"r": 5}, "float32"), (31, "generalized", "max", {"r": 5}, "float32"),
              (31, "generalized", "avg", {"r": 5}, "bfloat16"), (31, "generalized", "min", {"r": 5}, "int32"),
              (63, "generalized", "max", {"r": 6}, "float32"), (64, "rd", "max", {}, "float32"),
              (64, "rd", "max", {}, "bfloat16"), (31, "generalized", "sum", {"r": 3}, "float32"),
              (12, "generalized", "prod", {"r": 2}, "float32"), (31, "generalized", "max", {"r": 5}, "bfloat16"),
              (24, "generalized", "min", {"r": 4}, "bfloat16"),
              (17, "generalized", "sum", {"r": 2}, "float32")]


@pytest.mark.parametrize("P,algo,op,kw,dtype", WORD_CASES)
def test_compiled_dag_programs_of_many_inputs_bit_exact(P, algo, op, kw, dtype):
    """Rank-specific DAG programs at large P, compiled at run time: 17 to 32
    inputs on the staged kernel with consumers that take one 32-bit word of
    every staged tile per thread, more on the word kernel (one word of every
    rank buffer per thread, no staging), both evaluating the program level by
    level in registers (P = 12 keeps the 16-byte consumer; bf16 max / min go
    to the word kernel from 25 inputs): bit for bit the
    oracle's literal schedule, the ragged length's edges on the element-wise
    kernel, guard bands intact."""
    import collective_reduction_gb300 as ar
    n = 40_009 if P > 16 else 100_003
    dist = "uniform_int" if dtype == "int32" else "normal"
    bufs = ar_synth.rank_inputs(P, n, dtype, dist, sigma=1.0, seed=P + 101)
    plan = ar.Plan(P, n, dtype, op, algo, jit="on", **kw)
    k = plan.info()["kernels"]
    selects = dtype == "bfloat16" and op in ("max", "min")
    assert k & (ar.KERNEL_WORD_JIT if P > 32 or (selects and P >= 25) else ar.KERNEL_DAG_JIT), k
    plan.close()
    want = oracle.run(algo, bufs, Arith(op, dtype), **kw).bufs
    got = engine(bufs, dtype, op, algo, jit="on", **kw)
    for r in range(P):
        assert_bit_equal(got[r], want[r], dtype, f"{algo} {op} {kw} rank {r}")


@pytest.mark.parametrize("algo,kw", [("ring", {}), ("rh", {"form": "step"}), ("generalized", {"r": 3, "jit": "on"}),
                                     ("ring", {"order": "fp32acc"}), ("ring", {"phase": "all_gather"}),
                                     ("generalized", {"r": 3, "jit": "on", "P": 31}), ("rd", {"op": "max", "P": 40})])
def test_execute_captures_in_a_cuda_graph(algo, kw):
    """ar_execute only enqueues kernels: it can be captured in a CUDA graph
    whose replays give the same results as direct calls (the rank-streaming,
    step, compiled DAG, fp32-accumulate, copy, word-consumer and word
    kernels)."""
    import torch

    import collective_reduction_gb300 as ar
    kw = dict(kw)
    P, n, op = kw.pop("P", 7), (1 << 18) + 13, kw.pop("op", "sum")
    bufs = ar_synth.rank_inputs(P, n, "float32", "normal", sigma=1e-2, seed=23)
    plan = ar.Plan(P, n, "float32", op, algo, **kw)
    rd = RankBufs.from_host(bufs, "float32")
    direct = rd.views
    plan.execute(direct)
    torch.cuda.synchronize()
    rg = RankBufs.from_host(bufs, "float32")
    graphed = rg.views
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            plan.execute(graphed, stream=s)
    torch.cuda.synchronize()
    rg.fill(bufs)  # capture does not run the kernels: restore, replay once
    g.replay()
    torch.cuda.synchronize()
    plan.check()
    rd.check_guards("direct")
    rg.check_guards("graphed")
    for r in range(P):
        assert_bit_equal(to_host(graphed[r], "float32"), to_host(direct[r], "float32"), "float32", f"rank {r}")


def test_bounded_wait_gives_up_and_the_device_stays_usable():
    """A wait that nothing completes gives up after its limit, reports
    AR_ERR_TIMEOUT, and the next allreduce still runs correctly."""
    import time

    import collective_reduction_gb300 as ar
    t0 = time.perf_counter()
    assert ar.selftest_bounded_wait(200) == "AR_ERR_TIMEOUT"
    assert 0.19 <= time.perf_counter() - t0 < 5.0
    bufs = ar_synth.rank_inputs(4, 4099, "float32", "normal", seed=31)
    check_faithful(bufs, "float32", "sum", "ring", "fused")


@pytest.mark.parametrize("dtype", ["float32", "bfloat16", "int32"])
@pytest.mark.parametrize("op", ["sum", "prod"])
def test_two_rank_fp32acc_is_the_single_combine(dtype, op):
    """With two ranks the fp32 accumulation is one fp32 op and one rounding:
    the same bits as the order-faithful pass (which the plan then runs)."""
    dist = "small_int" if (dtype == "int32" and op == "prod") else ("uniform_int" if dtype == "int32" else "normal")
    bufs = ar_synth.rank_inputs(2, (1 << 20) + 7, dtype, dist, sigma=1.0, seed=5)
    want = engine(bufs, dtype, op, "ring")
    got = engine(bufs, dtype, op, "ring", order="fp32acc")
    for r in range(2):
        assert_bit_equal(got[r], want[r], dtype, f"rank {r}")
