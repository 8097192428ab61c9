"""Helpers shared by the GPU parity tests: run one problem through the C ABI
on torch CUDA buffers, run the oracle on the same storage, compare.

Comparison bound (the target's statement of parity):
  |D - ref| <= 2^-10 * (|alpha| * sum_k |a*b| + |beta*c| + |x_factor*x|)
             (+ one ulp of the output format at |ref| for 16-bit outputs),
  Y the same with alpha = 1 and no C or X term; bit-exact equality with the
  once-rounded oracle value on integer-valued inputs whose products and sums
  are exactly representable.

fp16 accumulator (rounded to fp16 once per tensor-core instruction, i.e.
after every chunk of 16 K for 16-bit inputs, 32 K for 8-bit): the
accumulator's error is at most
  E = (2^-11 * P + 2^-10 * sum_k |a*b|) / (1 - n * 2^-11),
P the oracle's sum over the n chunk boundaries of |exact running sum|; the
2^-11 * P term is half an fp16 ulp (relative) per rounding, the 2^-10 term
the fp32 path's own bound for the products inside an instruction, and the
divisor absorbs the rounding of already-rounded errors.  D's bound takes
|alpha| * E in place of 2^-10 * |alpha| * sum|ab|; Y's is E.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

import oracle
import workloads as W
import dense_gemm_epilogue_persistent_gb300 as G

TOL_REL = 2.0 ** -10
U16 = 2.0 ** -11                               # unit roundoff of fp16
ULP = {"f16": (10, -14), "bf16": (7, -126)}   # fraction bits, min normal exponent


def ulp_at(dtype: str, ref: np.ndarray) -> np.ndarray:
    """Spacing of the output format at |ref| (subnormal spacing below normal)."""
    if dtype not in ULP:
        return np.zeros_like(ref)
    mant, emin = ULP[dtype]
    a = np.abs(ref)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(np.where(a > 0, e, emin), emin)
    return np.exp2(e - mant)


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.double().cpu().numpy()


@dataclasses.dataclass
class Case:
    """One problem: logical inputs plus layout/type/scalar choices."""
    M: int
    N: int
    K: int
    L: int
    ab: str = "f16"
    c: str | None = "f32"
    d: str = "f32"
    x: str | None = None
    y: str | None = None
    a_mn: bool = False
    b_mn: bool = False
    cd_m: bool = False
    alpha: float = 1.0
    beta: float = 0.0
    xf: float = 0.0
    dist: str = "normal1"
    seed: int = 0
    lda_pad: int = 0
    ldb_pad: int = 0
    b: str | None = None      # B's type when it differs from A's (fp8 pairs)
    relu: bool = False
    acc: str = "f32"          # tensor-core accumulator

    @staticmethod
    def from_workload(w: W.Workload, **over):
        kw = dict(M=w.M, N=w.N, K=w.K, L=w.L, ab=w.ab, c=w.c, d=w.d, x=w.x, y=w.y,
                  a_mn=w.a_mn_major, b_mn=w.b_mn_major, cd_m=w.cd_m_major, alpha=w.alpha,
                  beta=w.beta, xf=w.x_factor, dist=w.dist, seed=w.seed, b=w.b, relu=w.relu,
                  acc=w.acc)
        kw.update(over)
        return Case(**kw)

    def workload(self) -> W.Workload:
        return W.Workload("case", self.M, self.N, self.K, self.L, self.ab, self.a_mn, self.b_mn,
                          self.c, self.d, self.x, self.y, self.cd_m, self.alpha, self.beta,
                          self.xf, self.seed, self.dist, self.b, self.relu, self.acc)

    @property
    def acc_chunk(self) -> int:
        """K per tensor-core instruction when the accumulator is fp16, else 0."""
        if self.acc != "f16":
            return 0
        return 32 if W.ELEM_BYTES[self.ab] == 1 else 16


def _pad_ld(t: torch.Tensor, pad: int) -> torch.Tensor:
    if pad == 0:
        return t
    junk = torch.full((*t.shape[:-1], pad), 3, dtype=t.dtype)
    return torch.cat([t, junk], dim=-1).contiguous()


@dataclasses.dataclass
class Prepared:
    case: Case
    inp: W.Inputs
    A: torch.Tensor      # CPU storage
    B: torch.Tensor
    C: torch.Tensor | None
    X: torch.Tensor | None


def prepare(case: Case, inputs: W.Inputs | None = None) -> Prepared:
    inp = inputs if inputs is not None else W.make_inputs(case.workload())
    A = _pad_ld(W.to_storage(inp.A, case.a_mn), case.lda_pad)
    B = _pad_ld(W.to_storage(inp.B, case.b_mn), case.ldb_pad)
    C = W.to_storage(inp.C, case.cd_m) if inp.C is not None else None
    X = W.to_storage(inp.X, case.cd_m) if inp.X is not None else None
    return Prepared(case, inp, A, B, C, X)


def out_shape(case: Case):
    return (case.L, case.N, case.M) if case.cd_m else (case.L, case.M, case.N)


def run_gpu(gemm: G.Gemm, prep: Prepared, stream=None, D=None, Y=None, use_x=True,
            C_dev=None, X_dev=None):
    """Copy storage to the GPU, call gemm_run, return (D, Y) device tensors."""
    c = prep.case
    dev = torch.device("cuda")
    A = prep.A.to(dev)
    B = prep.B.to(dev)
    C = C_dev if C_dev is not None else (prep.C.to(dev) if prep.C is not None else None)
    X = X_dev if X_dev is not None else (
        prep.X.to(dev) if (prep.X is not None and use_x) else None)
    if D is None:
        D = torch.empty(out_shape(c), dtype=W.TORCH_DTYPE[c.d], device=dev)
    if Y is None and c.y is not None:
        Y = torch.empty(out_shape(c), dtype=W.TORCH_DTYPE[c.y], device=dev)
    dt = G.make_dtypes(c.ab, c.c or "f32", c.d, c.x or "f32", c.y or "f32",
                       G.GEMM_MN_MAJOR if c.cd_m else G.GEMM_K_MAJOR, b=c.b,
                       epilogue=G.GEMM_EPI_RELU if c.relu else G.GEMM_EPI_LINEAR, acc=c.acc)
    gemm.run(c.M, c.N, c.K, c.L, A, A.shape[-1], int(c.a_mn), B, B.shape[-1], int(c.b_mn),
             C, X, D, Y, c.alpha, c.beta, c.xf, dt, stream)
    return D, Y


def oracle_problem(prep: Prepared, use_x=True) -> oracle.Problem:
    c = prep.case
    st = W.storage_view_np
    return oracle.Problem(c.M, c.N, c.K, c.L, st(prep.A), prep.A.shape[-1], c.a_mn,
                          st(prep.B), prep.B.shape[-1], c.b_mn,
                          st(prep.C) if prep.C is not None else None,
                          st(prep.X) if (prep.X is not None and use_x) else None,
                          c.ab, c.c or "f32", c.x or "f32", c.cd_m, c.alpha, c.beta, c.xf,
                          b_dtype=c.b, relu=c.relu, acc_chunk=c.acc_chunk)


def logical(t: torch.Tensor, cd_m: bool) -> torch.Tensor:
    """Device output in storage layout -> CPU logical [L, M, N]."""
    return W.from_storage(t.cpu(), cd_m)


def bound_acc(case: Case, S, P=None):
    """Bound on the accumulator's error (see the module docstring)."""
    if case.acc_chunk == 0:
        return TOL_REL * S
    n = -(-case.K // case.acc_chunk)
    assert n * U16 < 0.5, "K too long for the fp16-accumulator bound"
    return (U16 * P + TOL_REL * S) / (1.0 - n * U16)


def bound_D(case: Case, S, Cv, Xv, ref, P=None):
    b = abs(case.alpha) * bound_acc(case, S, P)
    if Cv is not None and case.beta != 0:
        b = b + TOL_REL * np.abs(case.beta * Cv)
    if Xv is not None and case.xf != 0:
        b = b + TOL_REL * np.abs(case.xf * Xv)
    return b + ulp_at(case.d, ref)


def assert_within(name, got, ref, bound):
    err = np.abs(got - ref)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{name}: {int(bad.sum())} of {bad.size} outside the bound; worst ratio "
            f"{float(np.nanmax(err / np.maximum(bound, 1e-300))):.3g}; first bad index "
            f"{idx.tolist()} got {got[bad][:5]} ref {ref[bad][:5]}")


def compare_full(prep: Prepared, D_dev, Y_dev, exact=False, use_x=True):
    """Element-by-element comparison of every output against the oracle."""
    c = prep.case
    D_ref, Y_ref, S, *rest = oracle.gemm(oracle_problem(prep, use_x))
    P = rest[0] if rest else None
    D = to_f64(logical(D_dev, c.cd_m))
    if exact:
        want = oracle.round_to(c.d, D_ref)
        want = want.astype(np.float64) if c.d == "f32" else oracle.decode(c.d, want).reshape(D.shape)
        np.testing.assert_array_equal(D, want)
    else:
        Cv = to_f64(prep.inp.C) if prep.inp.C is not None else None
        Xv = to_f64(prep.inp.X) if (prep.inp.X is not None and use_x) else None
        assert_within("D", D, D_ref, bound_D(c, S, Cv, Xv, D_ref, P))
    if Y_dev is not None:
        Y = to_f64(logical(Y_dev, c.cd_m))
        if exact:
            want = oracle.round_to(c.y, Y_ref)
            want = want.astype(np.float64) if c.y == "f32" else oracle.decode(c.y, want).reshape(Y.shape)
            np.testing.assert_array_equal(Y, want)
        else:
            assert_within("Y", Y, Y_ref, bound_acc(c, S, P) + ulp_at(c.y, Y_ref))
    return D_ref, Y_ref


def compare_sampled(prep: Prepared, D_dev, Y_dev, tile_m: int, tile_n: int, seed: int,
                    n_random=4096, full_lines=True):
    """Full-size check: seeded random entries plus whole rows and columns at
    tile boundaries, each computed one by one by the oracle."""
    c = prep.case
    p = oracle_problem(prep)
    ms, ns, ls, rows, cols = W.check_entries(c.M, c.N, c.L, tile_m, tile_n, seed, n_random)
    if full_lines:
        ls_all = range(c.L) if c.L <= 2 else sorted({0, c.L - 1})
        for l in ls_all:
            for r in rows:
                ms = np.concatenate([ms, np.full(c.N, r)])
                ns = np.concatenate([ns, np.arange(c.N)])
                ls = np.concatenate([ls, np.full(c.N, l)])
            for col in cols:
                ms = np.concatenate([ms, np.arange(c.M)])
                ns = np.concatenate([ns, np.full(c.M, col)])
                ls = np.concatenate([ls, np.full(c.M, l)])
    D_ref, Y_ref, S, *rest = oracle.gemm_entries(p, ms, ns, ls)
    P = rest[0] if rest else None
    Dl = logical(D_dev, c.cd_m)
    D = to_f64(Dl[ls, ms, ns])
    Cv = to_f64(prep.inp.C[ls, ms, ns]) if prep.inp.C is not None else None
    Xv = to_f64(prep.inp.X[ls, ms, ns]) if prep.inp.X is not None else None
    assert_within("D", D, D_ref, bound_D(c, S, Cv, Xv, D_ref, P))
    if Y_dev is not None:
        Y = to_f64(logical(Y_dev, c.cd_m)[ls, ms, ns])
        assert_within("Y", Y, Y_ref, bound_acc(c, S, P) + ulp_at(c.y, Y_ref))
    return len(ms)
