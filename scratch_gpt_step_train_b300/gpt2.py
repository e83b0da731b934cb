"""Thin ctypes binding of libgpt2b300 (the C-ABI in include/gpt2.h).

Argument marshalling only: every step of the training step runs in the CUDA
library.  PyTorch provides device memory (the workspace and token buffers) and
the CUDA stream.  There is no fallback: if the shared library is missing or
fails to load, constructing a model raises.
"""
import ctypes as ct
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libgpt2b300.so")

FP32, BF16 = 0, 1
# activation recompute flags, OR-ed into the mode
RECOMPUTE_GELU, RECOMPUTE_LN = 0x10, 0x20
# parameters only in bf16, stochastic rounding in AdamW (with BF16)
NO_MASTER = 0x40
ERRORS = {0: "OK", -1: "GPT2_ERR_ARG", -2: "GPT2_ERR_CUDA", -3: "GPT2_ERR_OOM",
          -4: "GPT2_ERR_STATE", -5: "GPT2_ERR_TOKEN_RANGE", -6: "GPT2_ERR_NONFINITE",
          -7: "GPT2_ERR_TIMEOUT", -8: "GPT2_ERR_IO"}

# name -> (restype, argtypes); every function declared in include/gpt2.h
_vp, _i, _f, _sz = ct.c_void_p, ct.c_int, ct.c_float, ct.c_size_t
_pf, _pi = ct.POINTER(ct.c_float), ct.POINTER(ct.c_int)
SIGNATURES = {
    "gpt2_workspace_bytes": (_sz, [_i] * 7),
    "gpt2_create": (_i, [ct.POINTER(_vp)] + [_i] * 6 + [ct.c_uint64, _i, _vp, _sz, _vp]),
    "gpt2_destroy": (None, [_vp]),
    "gpt2_last_error": (ct.c_char_p, [_vp]),
    "gpt2_set_stream": (_i, [_vp, _vp]),
    "gpt2_forward": (_i, [_vp, _vp, _vp, _pf]),
    "gpt2_forward_host": (_i, [_vp, _vp, _vp, _pf]),
    "gpt2_backward": (_i, [_vp]),
    "gpt2_adamw_step": (_i, [_vp] + [_f] * 6 + [_pf]),
    "gpt2_zero_grad": (_i, [_vp]),
    "gpt2_sync": (_i, [_vp]),
    "gpt2_num_params": (_sz, [_vp]),
    "gpt2_padded_vocab": (_i, [_vp]),
    "gpt2_get_params": (_i, [_vp, _pf]),
    "gpt2_set_params": (_i, [_vp, _pf]),
    "gpt2_get_grads": (_i, [_vp, _pf]),
    "gpt2_set_grads": (_i, [_vp, _pf]),
    "gpt2_get_opt_state": (_i, [_vp, _pf, _pf, _pi]),
    "gpt2_set_opt_state": (_i, [_vp, _pf, _pf, _i]),
    "gpt2_get_logits": (_i, [_vp, _pf]),
    "gpt2_get_loss": (_i, [_vp, _pf]),
    "gpt2_get_losses": (_i, [_vp, _pf]),
    "gpt2_grads_buffer": (_i, [_vp, ct.POINTER(_vp), ct.POINTER(_sz)]),
    "gpt2_params_buffer": (_i, [_vp, ct.POINTER(_vp), ct.POINTER(_vp), ct.POINTER(_sz)]),
    "gpt2_get_grad_count": (_i, [_vp, _pi]),
    "gpt2_set_grad_count": (_i, [_vp, _i]),
    "gpt2_adamw_step_shard": (_i, [_vp, _sz, _sz] + [_f] * 6 + [_pf]),
    "gpt2_set_grad_count_device": (_i, [_vp, _vp]),
    "gpt2_workspace_bytes_shard": (_sz, [_i] * 7 + [_sz, _sz]),
    "gpt2_create_shard": (_i, [ct.POINTER(_vp)] + [_i] * 6 + [ct.c_uint64, _i, _sz, _sz, _vp, _sz,
                                                             _vp]),
    "gpt2_shard_bounds": (_i, [_vp, ct.POINTER(_sz), ct.POINTER(_sz)]),
    "gpt2_get_shard_master": (_i, [_vp, _pf]),
    "gpt2_set_spike_skip": (_i, [_vp, _f, _f, _i]),
    "gpt2_last_step_info": (_i, [_vp, _pi, _pf, _pf]),
    "gpt2_save_checkpoint": (_i, [_vp, ct.c_char_p]),
    "gpt2_load_checkpoint": (_i, [_vp, ct.c_char_p]),
    "gpt2_prof_enable": (_i, [_vp, ct.c_uint]),
    "gpt2_launch_count": (ct.c_longlong, [_vp]),
    "gpt2_prof_reset": (_i, [_vp]),
    "gpt2_prof_num_classes": (_i, []),
    "gpt2_prof_name": (ct.c_char_p, [_i]),
    "gpt2_prof_read": (_i, [_vp, _i, ct.POINTER(ct.c_double), ct.POINTER(ct.c_longlong),
                            ct.POINTER(ct.c_double), ct.POINTER(ct.c_double)]),
}

_lib_handle = None


def lib():
    """Load libgpt2b300.so (raises if it is not built)."""
    global _lib_handle
    if _lib_handle is not None:
        return _lib_handle
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "`python -m scratch_gpt_step_train_b300.build`")
    h = ct.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        f = getattr(h, name)
        f.restype = res
        f.argtypes = args
    _lib_handle = h
    return h


class GPT2Error(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"{ERRORS.get(code, code)}: {msg}")
        self.code = code


def _fptr(a):
    return a.ctypes.data_as(_pf)


def padded_vocab(V):
    return ((V + 127) // 128) * 128


def workspace_bytes(L, H, C, V, T, B, mode=FP32, shard=None):
    if shard is None:
        return lib().gpt2_workspace_bytes(L, H, C, V, T, B, mode)
    return lib().gpt2_workspace_bytes_shard(L, H, C, V, T, B, mode, int(shard[0]), int(shard[1]))


class GPT2:
    """One GPT-2 model + optimizer state on the current CUDA device.  With
    shard=(lo, hi) the handle is one rank's ZeRO-1 handle: it holds the AdamW
    moments (and in bf16 mode the fp32 master) of the canonical slice
    [lo, hi) only (gpt2_create_shard)."""

    def __init__(self, L, H, C, V, T, B, seed=0, mode=FP32, stream=None, torch_workspace=True,
                 shard=None):
        import torch
        self.L, self.H, self.C, self.V, self.T, self.B = L, H, C, V, T, B
        self.mode = mode
        self._lib = lib()
        self._torch = torch
        if stream is None:
            stream = torch.cuda.current_stream()
        self.stream = stream
        nbytes = workspace_bytes(L, H, C, V, T, B, mode, shard)
        if nbytes == 0:
            raise GPT2Error(-1, f"shape rejected: L={L} H={H} C={C} V={V} T={T} B={B}")
        self._ws = None
        ws_ptr = None
        if torch_workspace:
            self._ws = torch.empty(nbytes + 256, dtype=torch.uint8, device="cuda")
            base = self._ws.data_ptr()
            ws_ptr = (base + 255) & ~255
        h = _vp()
        if shard is None:
            rc = self._lib.gpt2_create(ct.byref(h), L, H, C, V, T, B, seed, mode, ws_ptr,
                                       nbytes if ws_ptr else 0, stream.cuda_stream)
        else:
            rc = self._lib.gpt2_create_shard(ct.byref(h), L, H, C, V, T, B, seed, mode,
                                             int(shard[0]), int(shard[1]), ws_ptr,
                                             nbytes if ws_ptr else 0, stream.cuda_stream)
        if rc != 0:
            raise GPT2Error(rc, "gpt2_create failed")
        self.h = h
        self.n = self._lib.gpt2_num_params(h)
        lo, hi = _sz(), _sz()
        self._ck(self._lib.gpt2_shard_bounds(h, ct.byref(lo), ct.byref(hi)))
        self.shard = (lo.value, hi.value)
        self.n_state = hi.value - lo.value
        self.Vp = self._lib.gpt2_padded_vocab(h)
        self.workspace_bytes = nbytes

    def close(self):
        if getattr(self, "h", None):
            self._lib.gpt2_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _ck(self, rc):
        if rc != 0:
            msg = self._lib.gpt2_last_error(self.h)
            raise GPT2Error(rc, msg.decode() if msg else "")
        return rc

    # ---- training step -------------------------------------------------
    def forward(self, tokens, targets=None, sync_loss=False):
        """tokens/targets: int32 [B,T] CUDA tensors (or numpy arrays, copied through
        gpt2_forward_host).  Returns the loss if sync_loss, else None."""
        lossp = ct.c_float(0.0)
        lp = ct.byref(lossp) if sync_loss else None
        if isinstance(tokens, np.ndarray):
            tok = np.ascontiguousarray(tokens, dtype=np.int32)
            tgt = None if targets is None else np.ascontiguousarray(targets, dtype=np.int32)
            self._ck(self._lib.gpt2_forward_host(self.h, tok.ctypes.data,
                                                 None if tgt is None else tgt.ctypes.data, lp))
        else:
            assert tokens.dtype == self._torch.int32 and tokens.is_cuda and tokens.is_contiguous()
            tp = None
            if targets is not None:
                assert targets.dtype == self._torch.int32 and targets.is_contiguous()
                tp = targets.data_ptr()
            self._ck(self._lib.gpt2_forward(self.h, tokens.data_ptr(), tp, lp))
        return lossp.value if sync_loss else None

    def backward(self):
        self._ck(self._lib.gpt2_backward(self.h))

    def zero_grad(self):
        self._ck(self._lib.gpt2_zero_grad(self.h))

    def adamw_step(self, lr, b1=0.9, b2=0.95, eps=1e-8, wd=0.1, clip=1.0):
        norm = ct.c_float(0.0)
        self._ck(self._lib.gpt2_adamw_step(self.h, lr, b1, b2, eps, wd, clip, ct.byref(norm)))
        return norm.value

    def adamw_step_rc(self, lr, b1=0.9, b2=0.95, eps=1e-8, wd=0.1, clip=1.0):
        norm = ct.c_float(0.0)
        rc = self._lib.gpt2_adamw_step(self.h, lr, b1, b2, eps, wd, clip, ct.byref(norm))
        return rc, norm.value

    def sync(self):
        self._ck(self._lib.gpt2_sync(self.h))

    # ---- inspection ----------------------------------------------------
    def get_params(self):
        out = np.empty(self.n, np.float32)
        self._ck(self._lib.gpt2_get_params(self.h, _fptr(out)))
        return out

    def set_params(self, p):
        p = np.ascontiguousarray(p, dtype=np.float32)
        assert p.size == self.n
        self._ck(self._lib.gpt2_set_params(self.h, _fptr(p)))

    def get_grads(self):
        out = np.empty(self.n, np.float32)
        self._ck(self._lib.gpt2_get_grads(self.h, _fptr(out)))
        return out

    def set_grads(self, g):
        g = np.ascontiguousarray(g, dtype=np.float32)
        assert g.size == self.n
        self._ck(self._lib.gpt2_set_grads(self.h, _fptr(g)))

    def get_opt_state(self):
        """(m, v, t); m and v cover the handle's slice (all N on an unsharded handle)"""
        m = np.empty(self.n_state, np.float32)
        v = np.empty(self.n_state, np.float32)
        t = ct.c_int(0)
        self._ck(self._lib.gpt2_get_opt_state(self.h, _fptr(m), _fptr(v), ct.byref(t)))
        return m, v, t.value

    def set_opt_state(self, m, v, step):
        m = np.ascontiguousarray(m, dtype=np.float32)
        v = np.ascontiguousarray(v, dtype=np.float32)
        assert m.size == self.n_state and v.size == self.n_state
        self._ck(self._lib.gpt2_set_opt_state(self.h, _fptr(m), _fptr(v), int(step)))

    def get_shard_master(self):
        """the fp32 master of the handle's slice"""
        out = np.empty(self.n_state, np.float32)
        self._ck(self._lib.gpt2_get_shard_master(self.h, _fptr(out)))
        return out

    # ---- data parallelism (see dp.DataParallel) ----
    def _ws_view(self, ptr, nbytes, dtype):
        """torch view of device memory inside this handle's workspace"""
        if self._ws is None or not ptr:
            return None
        off = ptr - self._ws.data_ptr()
        assert 0 <= off and off + nbytes <= self._ws.numel()
        return self._ws[off:off + nbytes].view(dtype)

    def grads_tensor(self):
        """the fp32 gradient vector (canonical order) as a torch view"""
        p, n = _vp(), _sz()
        self._ck(self._lib.gpt2_grads_buffer(self.h, ct.byref(p), ct.byref(n)))
        return self._ws_view(p.value, n.value * 4, self._torch.float32)

    def param_tensors(self):
        """(fp32 master or None, bf16 compute copy or None) as torch views"""
        pm, pb, n = _vp(), _vp(), _sz()
        self._ck(self._lib.gpt2_params_buffer(self.h, ct.byref(pm), ct.byref(pb), ct.byref(n)))
        return (self._ws_view(pm.value, n.value * 4, self._torch.float32),
                self._ws_view(pb.value, n.value * 2, self._torch.bfloat16))

    def grad_count(self):
        c = ct.c_int(0)
        self._ck(self._lib.gpt2_get_grad_count(self.h, ct.byref(c)))
        return c.value

    def set_grad_count(self, count):
        self._ck(self._lib.gpt2_set_grad_count(self.h, int(count)))

    def set_grad_count_device(self, count):
        """the next update divides by the int32 in the CUDA tensor `count`"""
        assert count.dtype == self._torch.int32 and count.is_cuda
        self._count_ref = count  # kept alive until the update has read it
        self._ck(self._lib.gpt2_set_grad_count_device(self.h, count.data_ptr()))

    def adamw_step_shard(self, lo, hi, lr, b1=0.9, b2=0.95, eps=1e-8, wd=0.1, clip=1.0):
        norm = ct.c_float(0.0)
        self._ck(self._lib.gpt2_adamw_step_shard(self.h, int(lo), int(hi), lr, b1, b2, eps, wd,
                                                 clip, ct.byref(norm)))
        return norm.value

    def set_spike_skip(self, loss_z=5.0, grad_z=5.0, window=128):
        """Skip the update when the step's mean loss or gradient norm has a
        z-score above its threshold against the previous `window` steps
        (window 0: off)."""
        self._ck(self._lib.gpt2_set_spike_skip(self.h, float(loss_z), float(grad_z), int(window)))

    def last_step_info(self):
        """(skipped, z_loss, z_grad) of the last adamw_step"""
        sk = ct.c_int(0)
        zl = ct.c_float(0.0)
        zg = ct.c_float(0.0)
        self._ck(self._lib.gpt2_last_step_info(self.h, ct.byref(sk), ct.byref(zl), ct.byref(zg)))
        return bool(sk.value), zl.value, zg.value

    def save_checkpoint(self, path):
        self._ck(self._lib.gpt2_save_checkpoint(self.h, os.fsencode(path)))

    def load_checkpoint(self, path):
        self._ck(self._lib.gpt2_load_checkpoint(self.h, os.fsencode(path)))

    def get_logits(self):
        out = np.empty((self.B, self.T, self.V), np.float32)
        self._ck(self._lib.gpt2_get_logits(self.h, _fptr(out)))
        return out

    def get_loss(self):
        x = ct.c_float(0.0)
        self._ck(self._lib.gpt2_get_loss(self.h, ct.byref(x)))
        return x.value

    def get_losses(self):
        out = np.empty((self.B, self.T), np.float32)
        self._ck(self._lib.gpt2_get_losses(self.h, _fptr(out)))
        return out

    # ---- per-kernel event timing ---------------------------------------
    def prof_enable(self, classes=None):
        """time every class (classes=None), the named classes, or none ([])"""
        if classes is None:
            mask = 0xFFFFFFFF
        else:
            names = self.prof_names()
            mask = 0
            for c in classes:
                mask |= 1 << names.index(c)
        self._ck(self._lib.gpt2_prof_enable(self.h, mask))

    def prof_names(self):
        return [self._lib.gpt2_prof_name(c).decode()
                for c in range(self._lib.gpt2_prof_num_classes())]

    def launch_count(self):
        return self._lib.gpt2_launch_count(self.h)

    def prof_reset(self):
        self._ck(self._lib.gpt2_prof_reset(self.h))

    def prof_read(self):
        """{class name: (ms, launches, flops, bytes)}"""
        out = {}
        for c in range(self._lib.gpt2_prof_num_classes()):
            ms, n = ct.c_double(), ct.c_longlong()
            fl, by = ct.c_double(), ct.c_double()
            self._ck(self._lib.gpt2_prof_read(self.h, c, ct.byref(ms), ct.byref(n),
                                              ct.byref(fl), ct.byref(by)))
            out[self._lib.gpt2_prof_name(c).decode()] = (ms.value, n.value, fl.value, by.value)
        return out
