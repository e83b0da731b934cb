"""A float64 PyTorch-CPU GPT-2 built from library routines, used only to pin
the oracle: F.layer_norm, F.linear, F.scaled_dot_product_attention (causal),
F.gelu(approximate="tanh"), F.cross_entropy, autograd, torch.optim.AdamW.

The architecture is the pre-LN GPT-2 of "Karpathy's llm.c: understanding LLM
training from scratch in C/CUDA" (section "Code anatomy"), with the readings
stated in the oracle's header (eps 1e-5, tanh GELU, padded vocabulary with
pad logits left out of the softmax, tied classifier).
"""
import numpy as np
import torch
import torch.nn.functional as F

from oracle.pyoracle import DECAYED, TENSOR_NAMES


def to_torch(params: dict):
    return {k: torch.tensor(np.array(v), dtype=torch.float64, requires_grad=True)
            for k, v in params.items()}


def forward(p, tok, tgt, L, H, C, V):
    tok = torch.as_tensor(np.asarray(tok), dtype=torch.long)
    B, T = tok.shape
    hd = C // H
    x = p["wte"][tok] + p["wpe"][:T]
    for l in range(L):
        h = F.layer_norm(x, (C,), p["ln1w"][l], p["ln1b"][l], eps=1e-5)
        qkv = F.linear(h, p["qkvw"][l], p["qkvb"][l])
        q, k, v = qkv.split(C, dim=-1)
        q, k, v = (t.reshape(B, T, H, hd).transpose(1, 2) for t in (q, k, v))
        y = F.scaled_dot_product_attention(q, k, v, is_causal=True)
        y = y.transpose(1, 2).reshape(B, T, C)
        x = x + F.linear(y, p["projw"][l], p["projb"][l])
        h = F.layer_norm(x, (C,), p["ln2w"][l], p["ln2b"][l], eps=1e-5)
        h = F.gelu(F.linear(h, p["fcw"][l], p["fcb"][l]), approximate="tanh")
        x = x + F.linear(h, p["fcprojw"][l], p["fcprojb"][l])
    x = F.layer_norm(x, (C,), p["lnfw"], p["lnfb"], eps=1e-5)
    logits = F.linear(x, p["wte"])[..., :V]
    if tgt is None:
        return logits, None
    tgt = torch.as_tensor(np.asarray(tgt), dtype=torch.long)
    loss = F.cross_entropy(logits.reshape(-1, V), tgt.reshape(-1))
    return logits, loss


def make_optimizer(p, lr, b1, b2, eps, wd):
    groups = [{"params": [p[k] for k in TENSOR_NAMES if k in DECAYED], "weight_decay": wd},
              {"params": [p[k] for k in TENSOR_NAMES if k not in DECAYED], "weight_decay": 0.0}]
    return torch.optim.AdamW(groups, lr=lr, betas=(b1, b2), eps=eps, foreach=False)


def clip_and_step(p, opt, clip):
    """Global-norm clip with no epsilon (min(1, clip/n)), then the optimizer step."""
    grads = [p[k].grad for k in TENSOR_NAMES]
    norm = torch.linalg.vector_norm(torch.cat([g.reshape(-1) for g in grads]))
    if clip > 0 and norm > clip:
        for g in grads:
            g.mul_(clip / norm)
    opt.step()
    return float(norm)
