"""The plain definition of the allreduce result.  TEST INFRASTRUCTURE ONLY.

Allreduce delivers to every rank the elementwise combination of all P vectors
(A Generalization of the Allreduce Operation, introduction).  For integers the
four ops are exact modulo 2^32 and independent of order, so any schedule must
reproduce ``direct_int`` bit for bit.  For floats the schedules differ in
rounding order ("All-Reduce, in depth", Numerics and reproducibility); the
reference every float result is measured against is the float64 combination
``direct_f64`` of the same inputs, and ``normwise_rel_err`` is the error
measure used for reordered (fp32-accumulated) results.
"""

import numpy as np

from .elementops import bf16_to_f32


def direct_int(bufs, op):
    """Exact int32 reduction of the rank buffers (wrapping sum / prod)."""
    acc = np.asarray(bufs[0], dtype=np.int32).view(np.uint32).copy()
    for b in bufs[1:]:
        b = np.asarray(b, dtype=np.int32).view(np.uint32)
        if op == "sum":
            acc = acc + b
        elif op == "prod":
            acc = acc * b
        elif op == "max":
            acc = np.maximum(acc.view(np.int32), b.view(np.int32)).view(np.uint32)
        elif op == "min":
            acc = np.minimum(acc.view(np.int32), b.view(np.int32)).view(np.uint32)
        else:
            raise ValueError(op)
    return acc.view(np.int32)


def as_f64(buf, dtype):
    if dtype == "bfloat16":
        return bf16_to_f32(buf).astype(np.float64)
    return np.asarray(buf).astype(np.float64)


def direct_f64(bufs, op, dtype):
    """float64 reduction of the rank buffers, ranks taken in order 0..P-1
    (avg: the float64 sum divided by P)."""
    acc = as_f64(bufs[0], dtype)
    for b in bufs[1:]:
        v = as_f64(b, dtype)
        if op in ("sum", "avg"):
            acc = acc + v
        elif op == "prod":
            acc = acc * v
        elif op == "max":
            acc = np.maximum(acc, v)
        elif op == "min":
            acc = np.minimum(acc, v)
        else:
            raise ValueError(op)
    if op == "avg":
        acc = acc / len(bufs)
    return acc


def normwise_rel_err(y, ref):
    """||y - ref||_2 / ||ref||_2 over all elements (0 when both vanish)."""
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    num = np.linalg.norm(y - ref)
    if den == 0.0:
        return 0.0 if num == 0.0 else float("inf")
    return float(num / den)
