"""The element operation of the allreduce.  TEST INFRASTRUCTURE ONLY.

Allreduce combines the ranks' vectors elementwise with one associative
operator (A Generalization of the Allreduce Operation, introduction; the
elementwise vector operator of "還元演算子" (Reduction operator), binomial-tree
section).  The engine supports sum, prod, max and min over int32, fp32 and
bf16.  The receiver's own value is always the LEFT operand: the ring of
"All-Reduce, in depth" (The ring algorithm) adds the arriving chunk into the
receiver's copy, and the binomial tree of "還元演算子" computes
x_i <- x_i (+) x_{i+2^k} on the receiving unit i.

Arithmetic rules (the pages fix none of them; these are the plain IEEE / two's
complement readings):
  int32  sum and prod wrap modulo 2^32; max / min are exact.
  fp32   IEEE binary32 with round-to-nearest-even, subnormals kept.
  bf16   both operands widened to fp32 (exact), the op done in fp32, the
         result rounded to bf16 with round-to-nearest-even after EVERY op.
  max    a > b ? a : b   (ties, +-0 and NaN keep the right operand b)
  min    a < b ? a : b
  avg    the sum, then divided by the rank count P ("All-Reduce, in depth",
         The APIs: ncclAvg divides by N inside the collective).  Combines are
         sums; ``average`` divides a finished sum once: fp32 IEEE division
         with round-to-nearest-even; bf16 widened, divided in fp32, rounded to
         bf16.  Float types only.
bf16 values are held as uint16 bit patterns.
"""

import numpy as np

DTYPES = ("int32", "float32", "bfloat16")
OPS = ("sum", "prod", "max", "min", "avg")
ESIZE = {"int32": 4, "float32": 4, "bfloat16": 2}
NP_STORAGE = {"int32": np.int32, "float32": np.float32, "bfloat16": np.uint16}


def bf16_to_f32(u16):
    """Widen bf16 bit patterns to fp32 values (exact: bf16 is the top half)."""
    u = np.asarray(u16, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32)


def f32_to_bf16_rne(x):
    """Round fp32 values to bf16 bit patterns, round-to-nearest, ties-to-even.

    The 16 dropped bits are compared with half an ulp of the kept part: the
    kept part is incremented when they exceed the half, or equal it and the
    kept part is odd.  A carry out of the mantissa raises the exponent, which
    also turns the largest values into infinity, as rounding must.  NaN maps
    to a quiet NaN of the same sign.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    bits = x.view(np.uint32).astype(np.uint64)
    kept = bits >> np.uint64(16)
    dropped = bits & np.uint64(0xFFFF)
    half = np.uint64(0x8000)
    odd = kept & np.uint64(1)
    round_up = (dropped > half) | ((dropped == half) & (odd == np.uint64(1)))
    out = (kept + round_up.astype(np.uint64)).astype(np.uint32)
    nan = np.isnan(x)
    if nan.any():
        sign = (bits >> np.uint64(31)).astype(np.uint32) << np.uint32(15)
        out = np.where(nan, sign | np.uint32(0x7FC0), out)
    return out.astype(np.uint16)


class Arith:
    """Numeric element operation for one (op, dtype)."""

    symbolic = False

    def __init__(self, op, dtype):
        if op not in OPS:
            raise ValueError(f"unknown op {op!r}")
        if dtype not in DTYPES:
            raise ValueError(f"unknown dtype {dtype!r}")
        if op == "avg" and dtype == "int32":
            raise ValueError("avg is defined for the float types only")
        self.op = op
        self.dtype = dtype
        self.storage = NP_STORAGE[dtype]
        self.combines = 0  # element operations performed

    def _f32_op(self, a, b):
        with np.errstate(over="ignore", invalid="ignore", under="ignore"):
            return self._f32_op_raw(a, b)

    def _f32_op_raw(self, a, b):
        if self.op in ("sum", "avg"):
            return np.add(a, b, dtype=np.float32)
        if self.op == "prod":
            return np.multiply(a, b, dtype=np.float32)
        if self.op == "max":
            return np.where(a > b, a, b)
        return np.where(a < b, a, b)

    def combine(self, a, b):
        """a (+) b elementwise, a being the receiver's own value."""
        a = np.asarray(a, dtype=self.storage)
        b = np.asarray(b, dtype=self.storage)
        self.combines += a.size
        if self.dtype == "int32":
            if self.op == "sum":
                return (a.view(np.uint32) + b.view(np.uint32)).view(np.int32)
            if self.op == "prod":
                return (a.view(np.uint32) * b.view(np.uint32)).view(np.int32)
            if self.op == "max":
                return np.where(a > b, a, b)
            return np.where(a < b, a, b)
        if self.dtype == "float32":
            return self._f32_op(a, b)
        fa, fb = bf16_to_f32(a), bf16_to_f32(b)
        if self.op == "max":
            # selection is exact: keep the chosen bit pattern, nothing rounds
            return np.where(fa > fb, a, b)
        if self.op == "min":
            return np.where(fa < fb, a, b)
        return f32_to_bf16_rne(self._f32_op(fa, fb))

    def average(self, x, P):
        """A finished avg sum divided by the rank count P (see the module
        docstring); not counted as a combine."""
        x = np.asarray(x, dtype=self.storage)
        d = np.float32(P)
        with np.errstate(over="ignore", invalid="ignore", under="ignore", divide="ignore"):
            if self.dtype == "float32":
                return np.divide(x, d, dtype=np.float32)
            return f32_to_bf16_rne(np.divide(bf16_to_f32(x), d, dtype=np.float32))

    def empty(self, n):
        return np.zeros(n, dtype=self.storage)


class Symbolic:
    """Element 'operation' that records the reduction tree instead of a value.

    A leaf is the int rank whose contribution it is; a combine of a (receiver,
    left) and b (incoming, right) is the tuple (a, b).  Running a schedule on
    rank buffers filled with their own rank number yields, per element, the
    exact parenthesisation the schedule fixes.
    """

    symbolic = True
    storage = object

    def __init__(self):
        self.combines = 0
        self._pair = np.frompyfunc(lambda a, b: (a, b), 2, 1)

    def combine(self, a, b):
        a = np.asarray(a, dtype=object)
        b = np.asarray(b, dtype=object)
        self.combines += a.size
        out = self._pair(a, b)
        return np.asarray(out, dtype=object).reshape(a.shape)

    def empty(self, n):
        return np.empty(n, dtype=object)


def leaf_buffers(P, n):
    """Symbolic rank buffers: every element of rank r is the leaf r."""
    bufs = []
    for r in range(P):
        b = np.empty(n, dtype=object)
        b[:] = [r] * n
        bufs.append(b)
    return bufs


def tree_str(t):
    """Canonical text of a tree: leaves as rank numbers, '(a+b)' for a combine."""
    if isinstance(t, tuple):
        return "(" + tree_str(t[0]) + "+" + tree_str(t[1]) + ")"
    return str(int(t))


def tree_leaves(t):
    """Leaves of a tree in left-to-right order."""
    out = []
    stack = [t]
    while stack:
        x = stack.pop()
        if isinstance(x, tuple):
            stack.append(x[1])
            stack.append(x[0])
        else:
            out.append(int(x))
    return out
