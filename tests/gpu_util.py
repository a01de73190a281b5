"""Helpers shared by the GPU tests: move seeded host buffers to the device,
run the engine through its C ABI, compare bit patterns."""

import numpy as np

import collective_reduction_gb300 as ar


def ensure_built():
    import os
    if not os.path.exists(ar.LIB_PATH):
        from collective_reduction_gb300 import build
        build.build()
    return ar.lib()


def to_dev(a, dtype):
    import torch
    if dtype == "bfloat16":
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16).copy()).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(a).copy())
    return t.cuda()


def to_host(t, dtype):
    import torch
    if dtype == "bfloat16":
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def engine(bufs, dtype, op, algo, **params):
    """Run the allreduce on copies of host buffers; returns host results."""
    import torch
    P, n = len(bufs), len(bufs[0])
    dev = [to_dev(b, dtype) for b in bufs]
    plan = ar.Plan(P, n, dtype, op, algo, **params)
    plan.execute(dev)
    torch.cuda.synchronize()
    plan.check()
    out = [to_host(t, dtype) for t in dev]
    plan.close()
    return out


def bits(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return a
    return a.view(np.uint32)


def nan_mask(a, dtype):
    if dtype == "float32":
        return np.isnan(a)
    if dtype == "bfloat16":
        return ((a & 0x7F80) == 0x7F80) & ((a & 0x7F) != 0)
    return np.zeros(a.shape, bool)


def assert_bit_equal(got, want, dtype, what=""):
    got, want = np.asarray(got), np.asarray(want)
    assert got.shape == want.shape, what
    gn, wn = nan_mask(got, dtype), nan_mask(want, dtype)
    assert np.array_equal(gn, wn), f"NaN positions differ {what}"
    keep = ~gn
    g, w = bits(got)[keep], bits(want)[keep]
    if not np.array_equal(g, w):
        idx = np.nonzero(g != w)[0]
        raise AssertionError(f"{what}: {idx.size} of {g.size} elements differ; first at {idx[:5]}: "
                             f"got {g[idx[:5]]} want {w[idx[:5]]}")
