"""Thin ctypes binding of liblmce.so (argument marshalling only).

Every step of the micro-step runs in the library's CUDA kernels.  PyTorch is used
here only to name device memory (``data_ptr()``) and streams.  If the library is
missing this module raises; there is no CPU fallback.
"""

from __future__ import annotations

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "liblmce.so")
DEBUG_LIB_PATH = os.path.join(HERE, "liblmce_dbg.so")   # built with the device bounds checks

OK = 0
ERR_ARG = 1
ERR_ARCH = 2
ERR_CUDA = 3
ERR_BAD_TARGET = 4
ERR_NO_VALID = 5
ERR_NONFINITE = 6
ERR_STATE = 7
ERR_INTERNAL = 8

DTYPES = {"bf16": 0, "fp32": 1}
NORMS = {"global": 0, "micro_mean": 1}
PATHS = {"auto": 0, "simt": 1, "tcgen05": 2, "tcgen05_two_pass": 3, "tcgen05_recompute": 4}
PATH_NAMES = {v: k for k, v in PATHS.items()}
TORCH_DTYPES = {"bf16": torch.bfloat16, "fp32": torch.float32}

EXPORTS = ("lmce_create", "lmce_microstep", "lmce_finalize", "lmce_destroy", "lmce_status_string",
           "lmce_launch_count", "lmce_selected_path", "lmce_profile", "lmce_profile_read",
           "lmce_microstep_noalloc", "lmce_dw_sumsq", "lmce_adamw", "lmce_microstep_compact",
           "lmce_microstep_ln", "lmce_microstep_ln_compact", "lmce_test_stall_next_microstep", "lmce_clip_coef",
           "lmce_debug_bounds", "lmce_test_bounds_limit")

NOALLOC_MAX_N = 65536

KINDS = {"lse": 0, "finish": 1, "dW": 2, "dh": 3, "lse_dh": 4, "ln": 5, "compact": 6}


class Config(ctypes.Structure):
    _fields_ = [("C", ctypes.c_int64), ("V", ctypes.c_int64), ("max_N", ctypes.c_int64),
                ("dtype", ctypes.c_int32), ("ignore_id", ctypes.c_int32), ("norm", ctypes.c_int32),
                ("grad_accum_steps", ctypes.c_int32), ("path", ctypes.c_int32),
                ("flags", ctypes.c_int32)]

ACCUMULATE_FROM_START = 1   # Config.flags: the first micro-step adds to dW instead of writing it
COMPACT_VALID_ROWS = 2      # Config.flags: scratch for microstep_compact
FINAL_NORM = 4              # Config.flags: scratch for microstep_ln
LN_KINDS = {"layernorm": 0, "rmsnorm": 1}


class LmceError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: lmce status {status} ({status_string(status)})")
        self.status = status


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load liblmce.so (once) and declare its signatures; raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with grad_lmce_microstep_gb300.build.build()")
    L = ctypes.CDLL(path)
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    L.lmce_create.argtypes = [ctypes.POINTER(Config), vp, ctypes.POINTER(vp)]
    L.lmce_create.restype = i32
    L.lmce_microstep.argtypes = [vp, vp, vp, vp, i64, i64, vp, vp, vp]
    L.lmce_microstep.restype = i32
    L.lmce_microstep_compact.argtypes = [vp, vp, vp, vp, i64, i64, i64, vp, vp, vp]
    L.lmce_microstep_compact.restype = i32
    L.lmce_microstep_ln.argtypes = [vp, vp, vp, vp, i32, ctypes.c_float, vp, vp, i64, i64, vp, vp, vp, vp, vp]
    L.lmce_microstep_ln.restype = i32
    L.lmce_microstep_ln_compact.argtypes = [vp, vp, vp, vp, i32, ctypes.c_float, vp, vp, i64, i64, i64, vp, vp, vp,
                                            vp, vp]
    L.lmce_microstep_ln_compact.restype = i32
    L.lmce_finalize.argtypes = [vp, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(i64),
                                ctypes.POINTER(ctypes.c_double), vp]
    L.lmce_finalize.restype = i32
    L.lmce_dw_sumsq.argtypes = [vp, ctypes.POINTER(ctypes.c_double), vp]
    L.lmce_dw_sumsq.restype = i32
    f32 = ctypes.c_float
    L.lmce_adamw.argtypes = [vp, vp, vp, vp, vp, i64, f32, f32, f32, f32, f32, f32, vp]
    L.lmce_adamw.restype = i32
    L.lmce_destroy.argtypes = [vp]
    L.lmce_destroy.restype = i32
    L.lmce_status_string.argtypes = [i32]
    L.lmce_status_string.restype = ctypes.c_char_p
    L.lmce_launch_count.argtypes = [vp]
    L.lmce_launch_count.restype = i64
    L.lmce_selected_path.argtypes = [vp]
    L.lmce_selected_path.restype = i32
    L.lmce_profile.argtypes = [vp, i32]
    L.lmce_profile.restype = i32
    L.lmce_profile_read.argtypes = [vp, i32, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(i64)]
    L.lmce_profile_read.restype = i32
    L.lmce_microstep_noalloc.argtypes = [ctypes.POINTER(Config), vp, vp, vp, i64, i64, vp, vp, i32, vp, vp, vp, vp]
    L.lmce_microstep_noalloc.restype = i32
    L.lmce_clip_coef.argtypes = [ctypes.c_double, ctypes.c_double, ctypes.POINTER(ctypes.c_float)]
    L.lmce_clip_coef.restype = i32
    L.lmce_test_stall_next_microstep.argtypes = [vp, i64]
    L.lmce_test_stall_next_microstep.restype = i32
    L.lmce_debug_bounds.argtypes = []
    L.lmce_debug_bounds.restype = i32
    L.lmce_test_bounds_limit.argtypes = [vp, i64]
    L.lmce_test_bounds_limit.restype = i32
    _lib = L
    return L


def clip_coef(sumsq: float, max_norm: float = 1.0) -> float:
    """Global-norm clip coefficient for lmce_adamw's `clip` (lmce_clip_coef).

    sumsq is the sum of squares over every gradient of the model (lmce_dw_sumsq gives the tied
    matrix's share), as torch.nn.utils.clip_grad_norm_ computes it.
    """
    out = ctypes.c_float()
    st = load().lmce_clip_coef(float(sumsq), float(max_norm), ctypes.byref(out))
    if st != OK:
        raise LmceError(st, "lmce_clip_coef")
    return float(out.value)


def status_string(status: int) -> str:
    return load().lmce_status_string(int(status)).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check_dev(t, name, dtype=None, shape=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


class Lmce:
    """One handle: the fp32 dW accumulator of one optimizer step plus the library scratch.

    >>> L = Lmce(C, V, max_N, dW, dtype="bf16")           # dW: CUDA fp32 [V, C]
    >>> for h, y in micro_batches: L.microstep(h, W, y, global_valid=n_valid, dh=dh)
    >>> loss_sum, count, loss_mean = L.finalize()

    path: "auto" (tensor cores when the shape allows, with the stored-exponential dW pass when
    its max_N x V bf16 scratch fits, else the recomputing one), "tcgen05" (stored exponentials,
    an error if they do not fit), "tcgen05_recompute" (logits recomputed for dW, no N x V
    scratch), "tcgen05_two_pass" (a separate logsumexp pass) or "simt" (fp32 FFMA kernels).
    """

    def __init__(self, C: int, V: int, max_N: int, dW: torch.Tensor, dtype: str = "bf16",
                 ignore_id: int = -100, norm: str = "global", grad_accum_steps: int = 1,
                 path: str = "auto", accumulate_from_start: bool = False, compact: bool = False,
                 final_norm: bool = False):
        _check_dev(dW, "dW", torch.float32, (V, C))
        self.lib = load()
        self.C, self.V, self.max_N = int(C), int(V), int(max_N)
        self.dtype = dtype
        self.dW = dW
        cfg = Config(self.C, self.V, self.max_N, DTYPES[dtype], int(ignore_id), NORMS[norm],
                     int(grad_accum_steps), PATHS[path],
                     (ACCUMULATE_FROM_START if accumulate_from_start else 0) | (COMPACT_VALID_ROWS if compact else 0)
                     | (FINAL_NORM if final_norm else 0))
        h = ctypes.c_void_p()
        st = self.lib.lmce_create(ctypes.byref(cfg), _ptr(dW), ctypes.byref(h))
        if st != OK:
            raise LmceError(st, "lmce_create")
        self.handle = h

    @property
    def path(self) -> str:
        return PATH_NAMES[self.lib.lmce_selected_path(self.handle)]

    @property
    def launches(self) -> int:
        return int(self.lib.lmce_launch_count(self.handle))

    def microstep(self, hidden, W, targets, global_valid: int = 0, dh=None, row_loss=None,
                  stream=None, check: bool = True) -> int:
        """Enqueue one micro-step; returns the status (raises on error when check)."""
        N = int(targets.numel())
        tdt = TORCH_DTYPES[self.dtype]
        if N > 0:
            _check_dev(hidden, "hidden", tdt, (N, self.C))
            _check_dev(W, "W", tdt, (self.V, self.C))
            _check_dev(targets, "targets", torch.int32, (N,))
            _check_dev(dh, "dh", tdt, (N, self.C))
            if row_loss is not None:
                _check_dev(row_loss, "row_loss", torch.float32, (N,))
        st = self.lib.lmce_microstep(self.handle, _ptr(hidden), _ptr(W), _ptr(targets), N,
                                     int(global_valid), _ptr(dh), _ptr(row_loss), _stream(stream))
        if check and st != OK:
            raise LmceError(st, "lmce_microstep")
        return st

    def microstep_compact(self, hidden, W, targets, n_valid: int = -1, global_valid: int = 0, dh=None,
                          row_loss=None, stream=None, check: bool = True) -> int:
        """A micro-step over the rows with a target in [0, V) only (handle made with compact=True).

        n_valid: this micro-step's valid targets, or -1 to let the library count them (blocking).
        dh and row_loss get zeros on the ignored rows.
        """
        N = int(targets.numel())
        tdt = TORCH_DTYPES[self.dtype]
        if N > 0:
            _check_dev(hidden, "hidden", tdt, (N, self.C))
            _check_dev(W, "W", tdt, (self.V, self.C))
            _check_dev(targets, "targets", torch.int32, (N,))
            _check_dev(dh, "dh", tdt, (N, self.C))
            if row_loss is not None:
                _check_dev(row_loss, "row_loss", torch.float32, (N,))
        st = self.lib.lmce_microstep_compact(self.handle, _ptr(hidden), _ptr(W), _ptr(targets), N, int(n_valid),
                                             int(global_valid), _ptr(dh), _ptr(row_loss), _stream(stream))
        if check and st != OK:
            raise LmceError(st, "lmce_microstep_compact")
        return st

    def microstep_ln(self, x, gamma, beta, W, targets, global_valid: int = 0, dx=None, dgamma=None, dbeta=None,
                     kind: str = "layernorm", eps: float = 1e-5, row_loss=None, stream=None, check: bool = True,
                     n_valid=None) -> int:
        """A micro-step with ln_f in front (handle made with final_norm=True): h = ln_f(x) feeds the
        head, dx is written, dgamma / dbeta (fp32 [C]) are written or accumulated like dW.

        n_valid (an int, -1 = counted by the library): run over the valid rows only
        (lmce_microstep_ln_compact; the handle also needs compact=True).
        """
        N = int(targets.numel())
        tdt = TORCH_DTYPES[self.dtype]
        if gamma is None or dgamma is None:
            raise ValueError("gamma and dgamma are required")
        _check_dev(gamma, "gamma", torch.float32, (self.C,))
        _check_dev(dgamma, "dgamma", torch.float32, (self.C,))
        if beta is not None:
            _check_dev(beta, "beta", torch.float32, (self.C,))
        if dbeta is not None:
            _check_dev(dbeta, "dbeta", torch.float32, (self.C,))
        if N > 0:
            _check_dev(x, "x", tdt, (N, self.C))
            _check_dev(W, "W", tdt, (self.V, self.C))
            _check_dev(targets, "targets", torch.int32, (N,))
            _check_dev(dx, "dx", tdt, (N, self.C))
            if row_loss is not None:
                _check_dev(row_loss, "row_loss", torch.float32, (N,))
        if n_valid is None:
            st = self.lib.lmce_microstep_ln(self.handle, _ptr(x), _ptr(gamma), _ptr(beta), LN_KINDS[kind],
                                            float(eps), _ptr(W), _ptr(targets), N, int(global_valid), _ptr(dx),
                                            _ptr(dgamma), _ptr(dbeta), _ptr(row_loss), _stream(stream))
            what = "lmce_microstep_ln"
        else:
            st = self.lib.lmce_microstep_ln_compact(self.handle, _ptr(x), _ptr(gamma), _ptr(beta), LN_KINDS[kind],
                                                    float(eps), _ptr(W), _ptr(targets), N, int(n_valid),
                                                    int(global_valid), _ptr(dx), _ptr(dgamma), _ptr(dbeta),
                                                    _ptr(row_loss), _stream(stream))
            what = "lmce_microstep_ln_compact"
        if check and st != OK:
            raise LmceError(st, what)
        return st

    def finalize(self, stream=None, check: bool = True):
        """Wait for the step, return (loss_sum, valid_count, loss_mean) [, status if not check]."""
        ls = ctypes.c_double()
        cnt = ctypes.c_int64()
        mean = ctypes.c_double()
        st = self.lib.lmce_finalize(self.handle, ctypes.byref(ls), ctypes.byref(cnt), ctypes.byref(mean),
                                    _stream(stream))
        if check:
            if st != OK:
                raise LmceError(st, "lmce_finalize")
            return ls.value, cnt.value, mean.value
        return ls.value, cnt.value, mean.value, st

    def dw_sumsq(self, stream=None) -> float:
        """Sum of dW**2 over all elements, float64, fixed reduction order (waits for the stream)."""
        out = ctypes.c_double()
        st = self.lib.lmce_dw_sumsq(self.handle, ctypes.byref(out), _stream(stream))
        if st != OK:
            raise LmceError(st, "lmce_dw_sumsq")
        return out.value

    def adamw(self, p, m, v, step: int, lr: float, W_out=None, betas=(0.9, 0.95), eps: float = 1e-8,
              weight_decay: float = 0.1, clip: float = 1.0, stream=None):
        """One AdamW step on the master weights p with this handle's dW (enqueued, no wait).

        p, m, v: CUDA fp32 [V, C], updated in place (m = v = 0 before step 1); W_out: CUDA bf16
        [V, C] or None, receives p rounded to bf16; clip: the global-norm clip coefficient.
        """
        shape = (self.V, self.C)
        for t, name in ((p, "p"), (m, "m"), (v, "v")):
            _check_dev(t, name, torch.float32, shape)
        if W_out is not None:
            _check_dev(W_out, "W_out", torch.bfloat16, shape)
        st = self.lib.lmce_adamw(self.handle, _ptr(p), _ptr(m), _ptr(v), _ptr(W_out), int(step), float(lr),
                                 float(betas[0]), float(betas[1]), float(eps), float(weight_decay),
                                 float(clip), _stream(stream))
        if st != OK:
            raise LmceError(st, "lmce_adamw")

    def test_stall_next_microstep(self, wait_ns: int) -> int:
        """Failure-detection test hook: the next micro-step's tensor-core gradient launches start
        no load and give up after wait_ns (lmce_finalize then reports LMCE_ERR_CUDA)."""
        return int(self.lib.lmce_test_stall_next_microstep(self.handle, int(wait_ns)))

    def test_bounds_limit(self, rows: int) -> int:
        """Debug-build test hook: the compaction's bounds checks see `rows` compact rows
        (lmce_test_bounds_limit); the release build returns ERR_STATE."""
        return int(self.lib.lmce_test_bounds_limit(self.handle, int(rows)))

    def profile(self, enable: bool):
        """Record CUDA events around every kernel launch (enable=True clears old records)."""
        st = self.lib.lmce_profile(self.handle, 1 if enable else 0)
        if st != OK:
            raise LmceError(st, "lmce_profile")

    def profile_read(self):
        """{kind: (total_ms, launches)} of the recorded kernel launches."""
        out = {}
        for name, k in KINDS.items():
            ms = ctypes.c_double()
            n = ctypes.c_int64()
            st = self.lib.lmce_profile_read(self.handle, k, ctypes.byref(ms), ctypes.byref(n))
            if st != OK:
                raise LmceError(st, "lmce_profile_read")
            out[name] = (ms.value, n.value)
        return out

    def close(self):
        if getattr(self, "handle", None):
            self.lib.lmce_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *a):
        self.close()


def run_step(W, micro_batches, dtype: str, norm: str = "global", path: str = "auto", ignore_id: int = -100,
             row_loss: bool = False, dW=None, global_valid=None, compact: bool = False):
    """Convenience: one optimizer step over CUDA micro-batches [(h, y)].

    compact=True runs every micro-step over its valid rows only (lmce_microstep_compact).

    Returns (dW, [dh_k], [row_loss_k or None], (loss_sum, count, loss_mean, status)).
    """
    V, C = W.shape
    max_N = max([int(y.numel()) for _, y in micro_batches] + [1])
    if dW is None:
        dW = torch.empty(V, C, dtype=torch.float32, device=W.device)
    if global_valid is None:
        global_valid = sum(int(((y >= 0) & (y < V)).sum()) for _, y in micro_batches)
    L = Lmce(C, V, max_N, dW, dtype, ignore_id, norm, len(micro_batches), path, compact=compact)
    try:
        dhs, rls = [], []
        for h, y in micro_batches:
            dh = torch.empty_like(h)
            rl = torch.empty(y.numel(), dtype=torch.float32, device=W.device) if row_loss else None
            if compact:
                n_valid = int(((y >= 0) & (y < V)).sum())
                L.microstep_compact(h, W, y, n_valid, global_valid, dh, rl, check=False)
            else:
                L.microstep(h, W, y, global_valid, dh, rl, check=False)
            dhs.append(dh)
            rls.append(rl)
        res = L.finalize(check=False)
    finally:
        L.close()
    return dW, dhs, rls, res
