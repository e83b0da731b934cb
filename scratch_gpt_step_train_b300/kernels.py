"""ctypes binding of the kernel-level C-ABI (include/gpt2_kernels.h).

Each function takes torch CUDA tensors, checks dtypes / contiguity, and calls
the library; the work is enqueued on the current torch stream.  Argument
marshalling only.
"""
import ctypes as ct

from .gpt2 import GPT2Error, lib

_vp, _i, _l, _sz, _f = ct.c_void_p, ct.c_int, ct.c_long, ct.c_size_t, ct.c_float
SIGNATURES = {
    "gpt2k_binary_arch": (_i, []),
    "gpt2k_matmul_scratch_bytes": (_sz, []),
    "gpt2k_matmul": (_i, [_i, _i, _i, _i, _i, _vp, _l, _i, _vp, _l, _i, _vp, _l, _vp, _vp, _l,
                          _vp, _l, _i, _vp, _sz, _vp, _vp]),
    "gpt2k_matmul_bias_grad": (_i, [_i, _i, _i, _vp, _l, _i, _vp, _l, _i, _vp, _l, _vp, _l, _i,
                                    _vp, _vp, _sz, _vp, _vp]),
    "gpt2k_attention_forward": (_i, [_i, _vp, _vp, _vp, _i, _i, _i, _i, _vp]),
    "gpt2k_attention_backward_scratch_bytes": (_sz, [_i, _i, _i, _i]),
    "gpt2k_attention_backward": (_i, [_i, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp, _vp]),
    "gpt2k_layernorm_forward": (_i, [_i, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _vp]),
    "gpt2k_layernorm_backward_scratch_bytes": (_sz, [_i, _i]),
    "gpt2k_layernorm_backward": (_i, [_i, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i,
                                      _i, _vp, _vp]),
    "gpt2k_layernorm_backward_noalloc": (_i, [_i, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i,
                                              _i, _vp]),
    "gpt2k_encoder_forward": (_i, [_i, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp, _vp]),
    "gpt2k_encoder_backward_scratch_bytes": (_sz, [_i, _i, _i, _i]),
    "gpt2k_encoder_backward": (_i, [_i, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp, _vp]),
    "gpt2k_crossentropy": (_i, [_i, _vp, _vp, _vp, _i, _i, _i, _f, _vp, _vp]),
    "gpt2k_gelu_forward": (_i, [_i, _vp, _vp, _sz, _vp]),
    "gpt2k_stochastic_round_bf16": (_i, [_vp, _vp, _sz, ct.c_uint64, ct.c_uint64, _vp]),
    "gpt2k_bias_grad_scratch_bytes": (_sz, [_i, _i]),
    "gpt2k_bias_grad": (_i, [_i, _vp, _vp, _i, _i, _vp, _vp]),
}

EPI = {"store": 0, "gelu": 1, "resid": 2, "accum_f32": 3, "gelu_bwd": 4, "gelu_d": 5,
       "mul_aux": 6}
_bound = False


def klib():
    global _bound
    h = lib()
    if not _bound:
        for name, (res, args) in SIGNATURES.items():
            f = getattr(h, name)
            f.restype = res
            f.argtypes = args
        _bound = True
    return h


def _torch():
    import torch
    return torch


def _dt(t):
    torch = _torch()
    if t.dtype == torch.float32:
        return 0
    if t.dtype == torch.bfloat16:
        return 1
    raise TypeError(f"unsupported dtype {t.dtype}")


def _p(t):
    return None if t is None else t.data_ptr()


def _stream():
    return _torch().cuda.current_stream().cuda_stream


def _ck(rc, what):
    if rc != 0:
        raise GPT2Error(rc, what)


def _scratch(nbytes):
    torch = _torch()
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device="cuda")


def err_word():
    return _torch().zeros(4, dtype=_torch().int32, device="cuda")


def matmul(A, B, D, *, a_kmajor=True, b_kmajor=True, bias=None, resid=None, aux=None,
           epi="store", impl=0, err=None, M=None, N=None, K=None):
    """D[M,N] = epi(A . B^T); A is [M,K] (a_kmajor) or [K,M]; B is [N,K] or [K,N]."""
    L = klib()
    if M is None:
        M = A.shape[0] if a_kmajor else A.shape[1]
    if K is None:
        K = A.shape[1] if a_kmajor else A.shape[0]
    if N is None:
        N = B.shape[0] if b_kmajor else B.shape[1]
    for t in (A, B, D, bias, resid, aux):
        assert t is None or (t.is_cuda and t.is_contiguous())
    scratch = _scratch(L.gpt2k_matmul_scratch_bytes())
    err = err if err is not None else err_word()
    rc = L.gpt2k_matmul(_dt(A), impl, M, N, K, _p(A), A.shape[1], int(a_kmajor), _p(B),
                        B.shape[1], int(b_kmajor), _p(D), D.shape[1], _p(bias), _p(resid),
                        resid.shape[1] if resid is not None else 0, _p(aux),
                        aux.shape[1] if aux is not None else 0, EPI[epi], _p(scratch),
                        scratch.numel(), _p(err), _stream())
    _ck(rc, "gpt2k_matmul")
    return err


def matmul_bias_grad(A, B, D, aux, dbias, *, a_kmajor=True, b_kmajor=True, epi="mul_aux",
                     err=None):
    """D[M,N] = epi(A . B^T) (epi "mul_aux" or "gelu_bwd", bf16) and
    dbias[n] += sum_m D[m,n] (D's bf16 values summed in fp32)"""
    L = klib()
    M = A.shape[0] if a_kmajor else A.shape[1]
    K = A.shape[1] if a_kmajor else A.shape[0]
    N = B.shape[0] if b_kmajor else B.shape[1]
    for t in (A, B, D, aux, dbias):
        assert t.is_cuda and t.is_contiguous()
    scratch = _scratch(L.gpt2k_matmul_scratch_bytes())
    err = err if err is not None else err_word()
    rc = L.gpt2k_matmul_bias_grad(M, N, K, _p(A), A.shape[1], int(a_kmajor), _p(B), B.shape[1],
                                  int(b_kmajor), _p(D), D.shape[1], _p(aux), aux.shape[1],
                                  EPI[epi], _p(dbias), _p(scratch), scratch.numel(), _p(err),
                                  _stream())
    _ck(rc, "gpt2k_matmul_bias_grad")
    return err


def attention_forward(out, lse, qkv, B, T, C, H):
    _ck(klib().gpt2k_attention_forward(_dt(qkv), _p(out), _p(lse), _p(qkv), B, T, C, H,
                                       _stream()), "attention_forward")


def attention_backward(dqkv, dout, qkv, out, lse, B, T, C, H):
    L = klib()
    scratch = _scratch(L.gpt2k_attention_backward_scratch_bytes(B, T, C, H))
    _ck(L.gpt2k_attention_backward(_dt(qkv), _p(dqkv), _p(dout), _p(qkv), _p(out), _p(lse), B,
                                   T, C, H, _p(scratch), _stream()), "attention_backward")


def layernorm_forward(out, mean, rstd, x, w, b):
    N, C = x.shape
    _ck(klib().gpt2k_layernorm_forward(_dt(x), _p(out), _p(mean), _p(rstd), _p(x), _p(w), _p(b),
                                       N, C, _stream()), "layernorm_forward")


def layernorm_backward(dx, dw, db, dout, x, w, mean, rstd, dxsum=None, accumulate=True):
    L = klib()
    N, C = x.shape
    scratch = _scratch(L.gpt2k_layernorm_backward_scratch_bytes(N, C))
    _ck(L.gpt2k_layernorm_backward(_dt(x), _p(dx), _p(dw), _p(db), _p(dxsum), _p(dout), _p(x),
                                   _p(w), _p(mean), _p(rstd), N, C, int(accumulate), _p(scratch),
                                   _stream()), "layernorm_backward")


def layernorm_backward_noalloc(dx, dw, db, dout, x, w, mean, rstd):
    """As layernorm_backward, with the library's fixed device scratch instead
    of an allocation (for callers that cannot allocate; C <= 2048)."""
    N, C = x.shape
    rc = klib().gpt2k_layernorm_backward_noalloc(_dt(x), _p(dx), _p(dw), _p(db), _p(dout),
                                                 _p(x), _p(w), _p(mean), _p(rstd), N, C,
                                                 _stream())
    _ck(rc, "layernorm_backward_noalloc")


def encoder_forward(out, tok, wte, wpe, V, err=None):
    B, T = tok.shape
    C = wte.shape[1]
    err = err if err is not None else err_word()
    _ck(klib().gpt2k_encoder_forward(_dt(wte), _p(out), _p(tok), _p(wte), _p(wpe), B, T, C, V,
                                     _p(err), _stream()), "encoder_forward")
    return err


def encoder_backward(dwte, dwpe, dx, tok):
    L = klib()
    B, T = tok.shape
    Vp, C = dwte.shape
    scratch = _scratch(L.gpt2k_encoder_backward_scratch_bytes(B, T, C, Vp))
    _ck(L.gpt2k_encoder_backward(_dt(dx), _p(dwte), _p(dwpe), _p(dx), _p(tok), B, T, C, Vp,
                                 _p(scratch), _stream()), "encoder_backward")


def crossentropy(logits, losses, tgt, V, dloss, err=None):
    N, Vp = logits.shape
    err = err if err is not None else err_word()
    _ck(klib().gpt2k_crossentropy(_dt(logits), _p(logits), _p(losses), _p(tgt), N, V, Vp,
                                  float(dloss), _p(err), _stream()), "crossentropy")
    return err


def gelu_forward(out, inp):
    assert out.is_contiguous() and inp.is_contiguous() and out.numel() == inp.numel()
    _ck(klib().gpt2k_gelu_forward(_dt(inp), _p(out), _p(inp), inp.numel(), _stream()),
        "gelu_forward")


def stochastic_round_bf16(out, inp, seed, k0=0):
    """out (bf16) = stochastic rounding of inp (fp32) with stream counters k0.."""
    assert out.is_contiguous() and inp.is_contiguous() and out.numel() == inp.numel()
    _ck(klib().gpt2k_stochastic_round_bf16(_p(out), _p(inp), inp.numel(), int(seed), int(k0),
                                           _stream()), "stochastic_round_bf16")


def bias_grad(db, dout):
    L = klib()
    N, OC = dout.shape
    scratch = _scratch(L.gpt2k_bias_grad_scratch_bytes(N, OC))
    _ck(L.gpt2k_bias_grad(_dt(dout), _p(db), _p(dout), N, OC, _p(scratch), _stream()),
        "bias_grad")
