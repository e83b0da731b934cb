"""Parity of the linear-layer kernel (tcgen05 tensor cores, bf16 operands,
fp32 accumulation, fused epilogues) and of the fp32-FFMA kernel against the
oracle's matmul (fp64) on the same bf16-rounded inputs.

Element bound: |got - ref| <= (K 2^-24 + 1e-7) (|A| |B|^T) + 2^-8 |ref|, the
first term for fp32 accumulation in any order, the second for the final bf16
rounding (fp32 outputs drop it)."""
import numpy as np
import pytest
import torch

from oracle.pyoracle import Ops
from scratch_gpt_step_train_b300 import kernels as K

pytestmark = pytest.mark.gpu
ops = Ops("double")


def _bf(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).cuda()


def _np(t):
    return t.float().cpu().numpy().astype(np.float64)


def _operands(M, N, Kd, seed, a_kmajor, b_kmajor):
    rng = np.random.default_rng(seed)
    A = rng.normal(0, 1, (M, Kd))
    B = rng.normal(0, 1, (N, Kd)) * 0.05
    At = _bf(A if a_kmajor else A.T)
    Bt = _bf(B if b_kmajor else B.T)
    A64 = _np(At) if a_kmajor else _np(At).T
    B64 = _np(Bt) if b_kmajor else _np(Bt).T
    return At, Bt, np.ascontiguousarray(A64), np.ascontiguousarray(B64)


def _bound(A64, B64, ref, Kd, out_bf16=True, rows=None):
    a = np.abs(A64 if rows is None else A64[rows])
    absprod = ops.matmul_forward(a, np.abs(B64))
    b = (Kd * 2.0 ** -24 + 1e-7) * absprod
    if out_bf16:
        b = b + 2.0 ** -8 * np.abs(ref)
    return b + 1e-30


LAYOUTS = [(True, True), (True, False), (False, True), (False, False)]


@pytest.mark.parametrize("a_km,b_km", LAYOUTS, ids=["AK-BK", "AK-BN", "AM-BK", "AM-BN"])
@pytest.mark.parametrize("shape", [(296, 328, 200), (136, 8, 64), (64, 136, 8)],
                         ids=["ragged", "thin", "k8"])
@pytest.mark.parametrize("impl", [2, 1], ids=["tcgen05", "ffma"])
def test_matmul_store_bias(a_km, b_km, shape, impl):
    M, N, Kd = shape
    At, Bt, A64, B64 = _operands(M, N, Kd, 1, a_km, b_km)
    bias = _bf(np.random.default_rng(2).normal(0, 1, N))
    D = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    K.matmul(At, Bt, D, a_kmajor=a_km, b_kmajor=b_km, bias=bias, impl=impl, M=M, N=N, K=Kd)
    ref = ops.matmul_forward(A64, B64, _np(bias))
    got = _np(D)
    assert np.all(np.abs(got - ref) <= _bound(A64, B64, ref, Kd))


@pytest.mark.parametrize("a_km,b_km", LAYOUTS, ids=["AK-BK", "AK-BN", "AM-BK", "AM-BN"])
def test_matmul_epilogues(a_km, b_km):
    M, N, Kd = 296, 328, 200
    rng = np.random.default_rng(3)
    At, Bt, A64, B64 = _operands(M, N, Kd, 4, a_km, b_km)
    bias = _bf(rng.normal(0, 1, N))
    acc = ops.matmul_forward(A64, B64)
    bnd = _bound(A64, B64, acc, Kd, out_bf16=False)
    # GELU: aux = acc + bias, D = gelu(aux)
    D = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    aux = torch.empty_like(D)
    K.matmul(At, Bt, D, a_kmajor=a_km, b_kmajor=b_km, bias=bias, aux=aux, epi="gelu", impl=2,
             M=M, N=N, K=Kd)
    pre = acc + _np(bias)
    assert np.all(np.abs(_np(aux) - pre) <= bnd + 2.0 ** -8 * np.abs(pre))
    gl = ops.gelu_forward(pre)
    assert np.all(np.abs(_np(D) - gl) <= 1.2 * bnd + 2.0 ** -8 * np.abs(gl) + 1e-30)
    # residual: D = resid + acc + bias
    resid = _bf(rng.normal(0, 1, (M, N)))
    K.matmul(At, Bt, D, a_kmajor=a_km, b_kmajor=b_km, bias=bias, resid=resid, epi="resid",
             impl=2, M=M, N=N, K=Kd)
    ref = pre + _np(resid)
    assert np.all(np.abs(_np(D) - ref) <= bnd + 2.0 ** -8 * np.abs(ref))
    # GELU backward: D = acc * gelu'(aux)
    auxin = _bf(rng.normal(0, 1.5, (M, N)))
    K.matmul(At, Bt, D, a_kmajor=a_km, b_kmajor=b_km, aux=auxin, epi="gelu_bwd", impl=2,
             M=M, N=N, K=Kd)
    ref = ops.gelu_backward(_np(auxin), acc)
    gp = np.abs(ops.gelu_backward(_np(auxin), np.ones_like(acc)))
    # + fp32 evaluation of gelu': its two terms cancel near x = -0.75
    assert np.all(np.abs(_np(D) - ref) <= gp * bnd * 1.01 + 2.0 ** -8 * np.abs(ref)
                  + 4e-7 * np.abs(acc) + 1e-30)


# sup |gelu''| of the tanh-form GELU (attained at x = 0: 2 * 0.5 * sqrt(2/pi))
GELU2_SUP = 0.8


def test_gelu_second_derivative_bound():
    x = np.linspace(-8, 8, 160001)
    h = 1e-4
    g2 = (ops.gelu_backward(x + h, np.ones_like(x)) - ops.gelu_backward(x - h, np.ones_like(x))) / (2 * h)
    assert np.abs(g2).max() <= GELU2_SUP


@pytest.mark.parametrize("a_km,b_km", LAYOUTS, ids=["AK-BK", "AK-BN", "AM-BK", "AM-BN"])
@pytest.mark.parametrize("impl", [2, 1], ids=["tcgen05", "ffma"])
def test_matmul_gelu_derivative_epilogues(a_km, b_km, impl):
    """epi gelu_d: D = gelu(x), aux = gelu'(x) for x = acc + bias; epi mul_aux:
    D = acc * aux -- together the MLP's GELU forward and backward"""
    M, N, Kd = 296, 328, 200
    rng = np.random.default_rng(11)
    At, Bt, A64, B64 = _operands(M, N, Kd, 12, a_km, b_km)
    bias = _bf(rng.normal(0, 1, N))
    acc = ops.matmul_forward(A64, B64)
    bnd = _bound(A64, B64, acc, Kd, out_bf16=False)
    D = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    aux = torch.empty_like(D)
    K.matmul(At, Bt, D, a_kmajor=a_km, b_kmajor=b_km, bias=bias, aux=aux, epi="gelu_d",
             impl=impl, M=M, N=N, K=Kd)
    pre = acc + _np(bias)
    gl = ops.gelu_forward(pre)
    assert np.all(np.abs(_np(D) - gl) <= 1.2 * bnd + 2.0 ** -8 * np.abs(gl) + 1e-30)
    dg = ops.gelu_backward(pre, np.ones_like(pre))
    # |gelu'(x~) - gelu'(x)| <= sup|gelu''| |x~ - x|, plus the fp32 evaluation
    # of gelu' (its two terms cancel near x = -0.75) and the bf16 rounding
    assert np.all(np.abs(_np(aux) - dg) <= GELU2_SUP * bnd + 4e-7 + 2.0 ** -8 * np.abs(dg))
    auxin = _bf(rng.normal(0, 0.7, (M, N)))
    K.matmul(At, Bt, D, a_kmajor=a_km, b_kmajor=b_km, aux=auxin, epi="mul_aux", impl=impl,
             M=M, N=N, K=Kd)
    ref = acc * _np(auxin)
    assert np.all(np.abs(_np(D) - ref) <= np.abs(_np(auxin)) * bnd + 2.0 ** -8 * np.abs(ref)
                  + 1e-30)


@pytest.mark.parametrize("a_km,b_km", LAYOUTS, ids=["AK-BK", "AK-BN", "AM-BK", "AM-BN"])
@pytest.mark.parametrize("Kd", [200, 2000], ids=["nosplit", "splitK"])
def test_matmul_accumulate_fp32(a_km, b_km, Kd):
    """weight-gradient form: D (fp32) += A . B^T; K=2000 takes the split-K path"""
    M, N = 296, 328
    At, Bt, A64, B64 = _operands(M, N, Kd, 5, a_km, b_km)
    D0 = np.random.default_rng(6).normal(0, 1, (M, N)).astype(np.float32)
    D = torch.from_numpy(D0).cuda()
    K.matmul(At, Bt, D, a_kmajor=a_km, b_kmajor=b_km, epi="accum_f32", impl=2, M=M, N=N, K=Kd)
    acc = ops.matmul_forward(A64, B64)
    ref = D0.astype(np.float64) + acc
    bnd = _bound(A64, B64, acc, Kd, out_bf16=False) + 2.0 ** -24 * np.abs(ref)
    assert np.all(np.abs(D.cpu().numpy() - ref) <= bnd)
    # deterministic: the same call again gives the same bits
    D2 = torch.from_numpy(D0).cuda()
    K.matmul(At, Bt, D2, a_kmajor=a_km, b_kmajor=b_km, epi="accum_f32", impl=2, M=M, N=N, K=Kd)
    assert torch.equal(D, D2)


# Full-size products of the GPT-2 124M step at micro-batch 16 x 1024, as the
# bench runs them; the oracle computes a sample of 48 output rows (every
# column of each).
FULL = [
    ("qkv_fwd", 16384, 2304, 768, True, True, "store"),
    ("proj_fwd", 16384, 768, 768, True, True, "resid"),
    ("fc_fwd", 16384, 3072, 768, True, True, "gelu"),
    ("fcproj_fwd", 16384, 768, 3072, True, True, "resid"),
    ("classifier_fwd", 16384, 50304, 768, True, True, "store"),
    ("qkv_dx", 16384, 768, 2304, True, False, "store"),
    ("proj_dx", 16384, 768, 768, True, False, "store"),
    ("fc_dx", 16384, 768, 3072, True, False, "store"),
    ("fcproj_dx", 16384, 3072, 768, True, False, "gelu_bwd"),
    ("fc_fwd_gelu_d", 16384, 3072, 768, True, True, "gelu_d"),
    ("fcproj_dx_mul_aux", 16384, 3072, 768, True, False, "mul_aux"),
    ("classifier_dx", 16384, 768, 50304, True, False, "store"),
    ("qkv_dw", 2304, 768, 16384, False, False, "accum_f32"),
    ("proj_dw", 768, 768, 16384, False, False, "accum_f32"),
    ("fc_dw", 3072, 768, 16384, False, False, "accum_f32"),
    ("fcproj_dw", 768, 3072, 16384, False, False, "accum_f32"),
    ("classifier_dw", 50304, 768, 16384, False, False, "accum_f32"),
]


# The same products at the GPT-2 1558M width (C=1600, 3C=4800, 4C=6400; none a
# multiple of the 256-wide tiles) at micro-batch 16 x 1024.
FULL_1558M = [
    ("qkv_fwd", 16384, 4800, 1600, True, True, "store"),
    ("proj_fwd", 16384, 1600, 1600, True, True, "resid"),
    ("fc_fwd_gelu_d", 16384, 6400, 1600, True, True, "gelu_d"),
    ("fcproj_fwd", 16384, 1600, 6400, True, True, "resid"),
    ("classifier_fwd", 16384, 50304, 1600, True, True, "store"),
    ("qkv_dx", 16384, 1600, 4800, True, False, "store"),
    ("proj_dx", 16384, 1600, 1600, True, False, "store"),
    ("fc_dx", 16384, 1600, 6400, True, False, "store"),
    ("fcproj_dx_mul_aux", 16384, 6400, 1600, True, False, "mul_aux"),
    ("classifier_dx", 16384, 1600, 50304, True, False, "store"),
    ("qkv_dw", 4800, 1600, 16384, False, False, "accum_f32"),
    ("proj_dw", 1600, 1600, 16384, False, False, "accum_f32"),
    ("fc_dw", 6400, 1600, 16384, False, False, "accum_f32"),
    ("fcproj_dw", 1600, 6400, 16384, False, False, "accum_f32"),
    ("classifier_dw", 50304, 1600, 16384, False, False, "accum_f32"),
]

# The same products at the GPT-2 350M width (C=1024, 3C=3072, 4C=4096) at
# micro-batch 8 x 1024 (M = 8192 rows).
FULL_350M = [
    ("qkv_fwd", 8192, 3072, 1024, True, True, "store"),
    ("proj_fwd", 8192, 1024, 1024, True, True, "resid"),
    ("fc_fwd_gelu_d", 8192, 4096, 1024, True, True, "gelu_d"),
    ("fcproj_fwd", 8192, 1024, 4096, True, True, "resid"),
    ("classifier_fwd", 8192, 50304, 1024, True, True, "store"),
    ("qkv_dx", 8192, 1024, 3072, True, False, "store"),
    ("proj_dx", 8192, 1024, 1024, True, False, "store"),
    ("fc_dx", 8192, 1024, 4096, True, False, "store"),
    ("fcproj_dx_mul_aux", 8192, 4096, 1024, True, False, "mul_aux"),
    ("classifier_dx", 8192, 1024, 50304, True, False, "store"),
    ("qkv_dw", 3072, 1024, 8192, False, False, "accum_f32"),
    ("proj_dw", 1024, 1024, 8192, False, False, "accum_f32"),
    ("fc_dw", 4096, 1024, 8192, False, False, "accum_f32"),
    ("fcproj_dw", 1024, 4096, 8192, False, False, "accum_f32"),
    ("classifier_dw", 50304, 1024, 8192, False, False, "accum_f32"),
]
ALL_FULL = ([("124M-" + f[0],) + f[1:] for f in FULL]
            + [("1558M-" + f[0],) + f[1:] for f in FULL_1558M]
            + [("350M-" + f[0],) + f[1:] for f in FULL_350M])


@pytest.mark.parametrize("name,M,N,Kd,a_km,b_km,epi", ALL_FULL, ids=[f[0] for f in ALL_FULL])
def test_matmul_full_size_sampled(name, M, N, Kd, a_km, b_km, epi):
    g = torch.Generator(device="cuda").manual_seed(7)
    Ash = (M, Kd) if a_km else (Kd, M)
    Bsh = (N, Kd) if b_km else (Kd, N)
    At = torch.randn(Ash, generator=g, device="cuda").to(torch.bfloat16)
    Bt = (torch.randn(Bsh, generator=g, device="cuda") * 0.05).to(torch.bfloat16)
    bias = (torch.randn(N, generator=g, device="cuda")).to(torch.bfloat16)
    rows = np.sort(np.random.default_rng(8).choice(M, 48, replace=False))
    rt = torch.from_numpy(rows).cuda()
    A_rows = (At[rt] if a_km else At[:, rt].t()).float().cpu().numpy().astype(np.float64)
    B64 = (Bt if b_km else Bt.t()).float().cpu().numpy().astype(np.float64)
    acc = ops.matmul_forward(A_rows, B64)
    bnd = (Kd * 2.0 ** -24 + 1e-7) * ops.matmul_forward(np.abs(A_rows), np.abs(B64))
    if epi == "accum_f32":
        D = torch.zeros(M, N, device="cuda")
        K.matmul(At, Bt, D, a_kmajor=a_km, b_kmajor=b_km, epi=epi, impl=2, M=M, N=N, K=Kd)
        got = D[rt].cpu().numpy()
        assert np.all(np.abs(got - acc) <= bnd + 1e-30)
        return
    D = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    kw = {}
    ref = acc.copy()
    if epi in ("store", "gelu", "resid", "gelu_d"):
        kw["bias"] = bias
        ref = ref + _np(bias)
    if epi in ("gelu", "gelu_d"):
        kw["aux"] = torch.empty_like(D)
    if epi == "mul_aux":
        kw["aux"] = (torch.randn(M, N, generator=g, device="cuda") * 0.7).to(torch.bfloat16)
    if epi == "resid":
        kw["resid"] = torch.randn(M, N, generator=g, device="cuda").to(torch.bfloat16)
        ref = ref + _np(kw["resid"][rt])
    if epi == "gelu_bwd":
        kw["aux"] = torch.randn(M, N, generator=g, device="cuda").to(torch.bfloat16)
    K.matmul(At, Bt, D, a_kmajor=a_km, b_kmajor=b_km, epi=epi, impl=2, M=M, N=N, K=Kd, **kw)
    got = _np(D[rt])
    if epi == "gelu":
        assert np.all(np.abs(_np(kw["aux"][rt]) - ref) <= bnd + 2.0 ** -8 * np.abs(ref) + 1e-30)
        ref = ops.gelu_forward(ref)
        bnd = 1.2 * bnd
    if epi == "gelu_d":
        dg = ops.gelu_backward(ref, np.ones_like(ref))
        assert np.all(np.abs(_np(kw["aux"][rt]) - dg) <= GELU2_SUP * bnd + 4e-7
                      + 2.0 ** -8 * np.abs(dg))
        ref = ops.gelu_forward(ref)
        bnd = 1.2 * bnd
    if epi == "mul_aux":
        a = _np(kw["aux"][rt])
        ref = acc * a
        bnd = np.abs(a) * bnd
    if epi == "gelu_bwd":
        pre = _np(kw["aux"][rt])
        ref = ops.gelu_backward(pre, acc)
        bnd = np.abs(ops.gelu_backward(pre, np.ones_like(acc))) * bnd * 1.01 + 4e-7 * np.abs(acc)
    assert np.all(np.abs(got - ref) <= bnd + 2.0 ** -8 * np.abs(ref) + 1e-30)


# ------------------------------------------------ MLP input gradient + fc bias gradient

def _bias_grad_case(M, N, Kd, a_km, b_km, epi, seed):
    rng = np.random.default_rng(seed)
    At, Bt, A64, B64 = _operands(M, N, Kd, seed, a_km, b_km)
    aux = _bf(rng.normal(0, 0.7, (M, N)) if epi == "mul_aux" else rng.normal(0, 1.5, (M, N)))
    db0 = rng.normal(0, 1, N).astype(np.float32)
    D = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    db = torch.from_numpy(db0.copy()).cuda()
    K.matmul_bias_grad(At, Bt, D, aux, db, a_kmajor=a_km, b_kmajor=b_km, epi=epi)
    torch.cuda.synchronize()
    return At, Bt, A64, B64, aux, db0, D, db


@pytest.mark.parametrize("a_km,b_km", LAYOUTS, ids=["AK-BK", "AK-BN", "AM-BK", "AM-BN"])
@pytest.mark.parametrize("epi", ["mul_aux", "gelu_bwd"])
def test_matmul_bias_grad_against_the_oracle(a_km, b_km, epi):
    """D = acc * aux (or acc * gelu'(aux)) and dbias += sum over rows of D's
    bf16 values, at a size whose rows (1000: not a multiple of 32 or of the
    128-row tiles) and columns (392 against 256-wide tiles) are ragged.
    Bound on dbias: the sum over rows of each element's bound plus an fp32
    sum of M terms."""
    M, N, Kd = 1000, 392, 200
    At, Bt, A64, B64, aux, db0, D, db = _bias_grad_case(M, N, Kd, a_km, b_km, epi, 11)
    acc = ops.matmul_forward(A64, B64)
    bnd = _bound(A64, B64, acc, Kd, out_bf16=False)
    x = _np(aux)
    if epi == "mul_aux":
        ref = acc * x
        ebnd = np.abs(x) * bnd + 2.0 ** -24 * np.abs(ref)
    else:
        ref = ops.gelu_backward(x, acc)
        gp = np.abs(ops.gelu_backward(x, np.ones_like(acc)))
        ebnd = gp * bnd * 1.01 + 4e-7 * np.abs(acc) + 2.0 ** -24 * np.abs(ref)
    assert np.all(np.abs(_np(D) - ref) <= ebnd + 2.0 ** -8 * np.abs(ref) + 1e-30)
    want = db0.astype(np.float64) + ref.sum(axis=0)
    tol = ((ebnd + 2.0 ** -8 * np.abs(ref)).sum(axis=0)
           + (M + 2) * 2.0 ** -24 * (1.01 * np.abs(ref).sum(axis=0) + np.abs(db0)) + 1e-30)
    got = db.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - want) <= tol), np.max(np.abs(got - want) / tol)


@pytest.mark.parametrize("C", [768, 1600], ids=["124M", "1558M"])
def test_matmul_bias_grad_full_size(C):
    """the fcproj input gradient of a micro-batch of 16 x 1024 (A = dres
    [BT, C] K-major, B = W_fcproj stored [C, 4C]): dbias against the fp64 sum
    of D's bf16 values (the values the kernel sums), to an fp32 sum's error"""
    M, N, Kd = 16384, 4 * C, C
    At, Bt, A64, B64, aux, db0, D, db = _bias_grad_case(M, N, Kd, True, False, "mul_aux", 12)
    Dd = D.double()
    want = torch.from_numpy(db0).cuda().double() + Dd.sum(dim=0)
    tol = (M + 2) * 2.0 ** -24 * (Dd.abs().sum(dim=0) + abs(torch.from_numpy(db0).cuda().double())) + 1e-30
    assert bool(((db.double() - want).abs() <= tol).all())
    # and D itself on sampled rows against the oracle
    rows = np.sort(np.random.default_rng(13).choice(M, 24, replace=False))
    acc = ops.matmul_forward(A64[rows], B64)
    x = _np(aux[torch.from_numpy(rows).cuda()])
    ref = acc * x
    bnd = np.abs(x) * _bound(A64, B64, acc, Kd, out_bf16=False, rows=rows)
    assert np.all(np.abs(_np(D[torch.from_numpy(rows).cuda()]) - ref)
                  <= bnd + 2.0 ** -8 * np.abs(ref) + 1e-30)
