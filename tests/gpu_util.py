"""Helpers for the GPU parity tests: run a product through the C ABI and
compare it with the oracle element by element.

Bars (stated once, used by every GPU test):
* Boolean and tropical: bit-exact (uint32 views compared).
* plus-times fp32: |y - y_ref| <= 1e-5 * sum_j |A_ij x_j| + 1e-6, with y_ref
  and the scale sum accumulated in fp64 by the oracle.
"""
import numpy as np

import oracle
from oracle import BOOLEAN, PLUS_TIMES, RIGHT

PT_REL, PT_ABS = 1e-5, 1e-6


def torch_mod():
    import torch
    return torch


def device_product(tree, direction, semiring, x_np, B, w=1.0, n_in=None, n_out=None):
    """Run tree.spmv on device copies of x_np; return y as numpy."""
    torch = torch_mod()
    n_in = n_in if n_in is not None else (tree.n_cols if direction == RIGHT else tree.n_rows)
    n_out = n_out if n_out is not None else (tree.n_rows if direction == RIGHT else tree.n_cols)
    if semiring == BOOLEAN:
        x = torch.from_numpy(np.ascontiguousarray(x_np, np.uint32).view(np.int32).reshape(n_in)).cuda()
        y = torch.full((n_out,), -1, dtype=torch.int32, device="cuda")  # garbage: must be overwritten
    else:
        x = torch.from_numpy(np.ascontiguousarray(x_np, np.float32).reshape(n_in, B)).cuda()
        y = torch.full((n_out, B), float("nan"), dtype=torch.float32, device="cuda")
    tree.spmv(direction, semiring, x, y, B=B, w=w)
    torch.cuda.synchronize()
    out = y.cpu().numpy()
    return out.view(np.uint32) if semiring == BOOLEAN else out


def assert_match(semiring, got, ref: "oracle.OracleResult", where=""):
    if semiring == PLUS_TIMES:
        tol = oracle.plus_times_tolerance(ref.scale)
        err = np.abs(got.astype(np.float64) - ref.y)
        bad = ~(err <= tol)
        assert not bad.any(), "%s: %d of %d entries off, worst %g (tol %g)" % (
            where, int(bad.sum()), bad.size, float(err[bad].max()), float(tol[bad].max()))
    else:
        g = np.ascontiguousarray(got).view(np.uint32)
        r = np.ascontiguousarray(ref.y).view(np.uint32)
        bad = g != r
        assert not bad.any(), "%s: %d of %d entries differ" % (where, int(bad.sum()), bad.size)


def random_x(rng, semiring, n, B):
    if semiring == BOOLEAN:
        return rng.integers(0, 2 ** 32, size=n, dtype=np.uint64).astype(np.uint32)
    x = rng.uniform(-2, 2, size=(n, B)).astype(np.float32)
    if semiring == 2:
        x[rng.random(size=(n, B)) < 0.4] = np.inf
    return x
