"""Python binding of the layer-sliding fine-tuning library (include/sf.h).

Argument marshalling only: every step of the training path runs in the CUDA
library ``libsfslide.so`` built from ``csrc/``.  There is no fallback: if the
library is missing or fails to load, importing ``lib()`` raises.

Model API: ``Model`` wraps sf_init_model / sf_load_layer_weights /
sf_train_step / sf_get_grads / sf_loss.  Kernel API: the ``op_*`` functions
take device pointers (ints, e.g. ``tensor.data_ptr()``) and a stream handle.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np

from ._build import LIB as LIB_PATH, build  # noqa: F401

SF_OK, SF_EINVAL, SF_ENOMEM, SF_ECUDA, SF_ETIMEOUT, SF_ESTATE, SF_EDEVICE = 0, -1, -2, -3, -4, -5, -6
UNIT_EMBED, UNIT_FINAL_NORM, UNIT_LM_HEAD = -1, -2, -3
IGNORE_INDEX = -100
STATUS_NAMES = {0: "SF_OK", -1: "SF_EINVAL", -2: "SF_ENOMEM", -3: "SF_ECUDA",
                -4: "SF_ETIMEOUT", -5: "SF_ESTATE", -6: "SF_EDEVICE"}

# GEMM layouts and epilogues of sf_op_gemm
NT, NN, TN = 0, 1, 2
EPI_BF16, EPI_F32, EPI_F32_ADD, EPI_F32_ACC = 0, 1, 2, 3


class SfError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("n_layers", "hidden", "n_heads", "n_kv_heads", "head_dim", "ffn", "vocab",
                 "max_batch", "max_seq", "ring_slots", "lce_chunk_rows", "retain_grads")] + \
               [("rms_eps", ctypes.c_float), ("rope_base", ctypes.c_float),
                ("device", ctypes.c_int32), ("adam_threads", ctypes.c_int32),
                ("wait_timeout_ms", ctypes.c_int32), ("async_update", ctypes.c_int32),
                ("offload_activations", ctypes.c_int32), ("deterministic", ctypes.c_int32),
                ("qkv_bias", ctypes.c_int32), ("tie_embeddings", ctypes.c_int32),
                ("bf16_adam_state", ctypes.c_int32), ("fp16_grads", ctypes.c_int32),
                ("loss_scale", ctypes.c_float)]


class Adam(ctypes.Structure):
    _fields_ = [(n, ctypes.c_float) for n in ("lr", "beta1", "beta2", "eps", "weight_decay")]


class Stats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_double) for n in
                ("step_ms", "gemm_ms", "gemm_flops", "attn_ms", "attn_flops", "h2d_bytes",
                 "d2h_bytes", "host_adam_ms", "host_wait_ms")] + \
               [("gemm_launches", ctypes.c_int64), ("kernel_launches", ctypes.c_int64),
                ("timing_enabled", ctypes.c_int32)] + \
               [(n, ctypes.c_double) for n in
                ("fwd_layer_ms", "bwd_layer_ms", "d2h_layer_ms", "update_layer_ms", "loss_scale")] + \
               [("skipped_updates", ctypes.c_int64)] + \
               [(n, ctypes.c_double) for n in ("head_ms", "compute_ms", "exposed_ms")]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


class TraceEvent(ctypes.Structure):
    _fields_ = [("t_ms", ctypes.c_double), ("kind", ctypes.c_int32), ("unit", ctypes.c_int32)]


TRACE_KINDS = {1: "step_begin", 2: "gathered", 3: "wait_unit_begin", 4: "wait_unit_end",
               5: "update_begin", 6: "update_end", 7: "gpu_done", 8: "step_return"}

_lib = None

_VP, _I32, _I64, _F32, _SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
_SIGS = {
    "sf_unit_numel": (_SZ, [ctypes.POINTER(Config), _I32]),
    "sf_init_model": (ctypes.c_int, [ctypes.POINTER(Config), ctypes.POINTER(_VP)]),
    "sf_free": (None, [_VP]),
    "sf_last_error": (ctypes.c_char_p, [_VP]),
    "sf_load_layer_weights": (ctypes.c_int, [_VP, _I32, _VP, _SZ]),
    "sf_train_step": (ctypes.c_int, [_VP, _VP, _VP, _I32, _I32, ctypes.POINTER(Adam)]),
    "sf_train_step_accum": (ctypes.c_int, [_VP, _VP, _VP, _I32, _I32, _I32, ctypes.POINTER(Adam)]),
    "sf_get_grads": (ctypes.c_int, [_VP, _I32, _VP, _SZ]),
    "sf_get_weights": (ctypes.c_int, [_VP, _I32, _VP, _SZ]),
    "sf_get_adam_state": (ctypes.c_int, [_VP, _I32, _VP, _VP, _SZ]),
    "sf_set_adam_state": (ctypes.c_int, [_VP, _I32, _VP, _VP, _SZ]),
    "sf_get_adam_step": (ctypes.c_int, [_VP, ctypes.POINTER(_I64)]),
    "sf_set_adam_step": (ctypes.c_int, [_VP, _I64]),
    "sf_loss": (ctypes.c_int, [_VP, ctypes.POINTER(_F32)]),
    "sf_lce_step": (ctypes.c_int, [_VP, _VP, _VP, _VP, _I64, _I32, _I32, _I32, _VP, _VP, _VP]),
    "sf_sync": (ctypes.c_int, [_VP]),
    "sf_set_timing": (ctypes.c_int, [_VP, _I32]),
    "sf_get_stats": (ctypes.c_int, [_VP, ctypes.POINTER(Stats)]),
    "sf_debug_inject": (ctypes.c_int, [_VP, _I32, _I32]),
    "sf_get_trace": (ctypes.c_int, [_VP, ctypes.POINTER(TraceEvent), _I32, ctypes.POINTER(_I32)]),
    "sf_probe_host_bandwidth": (ctypes.c_int, [_I32, _I64, ctypes.POINTER(ctypes.c_double)]),
    "sf_op_gemm": (ctypes.c_int, [_I32, _I32, _I64, _I64, _I64, _VP, _I64, _VP, _I64, _VP, _I64,
                                  _VP, _I64, _F32, _VP]),
    "sf_op_rmsnorm_fwd": (ctypes.c_int, [_VP, _VP, _VP, _VP, _I64, _I32, _F32, _VP]),
    "sf_op_rmsnorm_bwd": (ctypes.c_int, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _I64, _I32, _VP]),
    "sf_op_rmsnorm_bwd_scratch": (_I64, [_I64, _I32]),
    "sf_op_rmsnorm_bwd_noalloc": (ctypes.c_int, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _I64, _I32, _VP]),
    "sf_rope_table": (ctypes.c_int, [_I32, _I32, _F32, _VP]),
    "sf_op_rope": (ctypes.c_int, [_VP, _I64, _I64, _I32, _I32, _I32, _VP, _I32, _VP]),
    "sf_op_gemm_qkv": (ctypes.c_int, [_I64, _I64, _I64, _VP, _I64, _VP, _I64, _VP, _I64, _VP, _VP,
                                      _I32, _I32, _I32, _VP]),
    "sf_op_gemm_swiglu": (ctypes.c_int, [_I64, _I64, _I64, _VP, _I64, _VP, _I64, _VP, _I64, _VP,
                                         _I64, _VP]),
    "sf_op_gemm_swiglu_bwd": (ctypes.c_int, [_I64, _I64, _I64, _VP, _I64, _VP, _I64, _VP, _I64,
                                             _VP, _I64, _VP]),
    "sf_op_gemm_bias": (ctypes.c_int, [_I64, _I64, _I64, _VP, _I64, _VP, _I64, _VP, _I64, _VP,
                                       ctypes.c_float, _VP]),
    "sf_op_bias_grad": (ctypes.c_int, [_VP, _I64, _I64, _I32, _VP, _VP, _VP]),
    "sf_op_bias_grad_scratch": (ctypes.c_int64, [_I64, _I32]),
    "sf_op_attn_fwd": (ctypes.c_int, [_VP, _VP, _VP, _I32, _I32, _I32, _I32, _I32, _VP]),
    "sf_op_attn_bwd": (ctypes.c_int, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _I32, _I32, _I32, _I32,
                                      _I32, _VP, _I32, _VP]),
    "sf_op_swiglu_fwd": (ctypes.c_int, [_VP, _VP, _I64, _I32, _VP]),
    "sf_op_swiglu_bwd": (ctypes.c_int, [_VP, _VP, _VP, _I64, _I32, _VP]),
    "sf_op_lce": (ctypes.c_int, [_VP, _VP, _VP, _I64, _I32, _I32, _I64, _I64, _VP, _VP, _VP, _VP, _VP]),
    "sf_op_lce_workspace_bytes": (_I64, [_I64, _I32, _I64]),
    "sf_op_lce_launches": (_I64, []),
    "sf_op_device_error": (ctypes.c_int, [ctypes.POINTER(_I32)]),
}


def exported_names():
    """Names declared by the C ABI (include/sf.h) that this binding wraps."""
    return list(_SIGS)


def lib(build_if_needed: bool = False) -> ctypes.CDLL:
    """Load libsfslide.so.  Raises if it does not exist (no fallback path)."""
    global _lib
    if _lib is None:
        if build_if_needed:
            build()
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "offloaded_fine_tuning_gb300.build() (needs nvcc)")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _check(st: int, ctx=None, what=""):
    if st != SF_OK:
        msg = lib().sf_last_error(ctx).decode(errors="replace") if ctx is not None or st != SF_EINVAL else ""
        raise SfError(st, f"{what}: {msg}")


def make_config(shape, max_batch=None, max_seq=None, ring_slots=None, retain_grads=1,
                lce_chunk_rows=0, device=0, adam_threads=0, wait_timeout_ms=0,
                async_update=0, offload_activations=0, deterministic=0,
                bf16_adam_state=0, fp16_grads=0, loss_scale=0.0) -> Config:
    """sf_config from a shape object with the fields of inputs.ModelConfig."""
    return Config(n_layers=shape.n_layers, hidden=shape.hidden, n_heads=shape.n_heads,
                  n_kv_heads=shape.n_kv_heads, head_dim=shape.head_dim, ffn=shape.ffn,
                  vocab=shape.vocab, max_batch=max_batch or shape.batch,
                  max_seq=max_seq or shape.seq,
                  ring_slots=ring_slots or shape.ring_slots, lce_chunk_rows=lce_chunk_rows,
                  retain_grads=retain_grads, rms_eps=shape.rms_eps, rope_base=shape.rope_base,
                  device=device, adam_threads=adam_threads, wait_timeout_ms=wait_timeout_ms,
                  async_update=async_update, offload_activations=offload_activations,
                  deterministic=deterministic,
                  qkv_bias=int(getattr(shape, "qkv_bias", False)),
                  tie_embeddings=int(getattr(shape, "tie_embeddings", False)),
                  bf16_adam_state=bf16_adam_state, fp16_grads=fp16_grads,
                  loss_scale=loss_scale)


def unit_numel(cfg: Config, unit: int) -> int:
    return int(lib().sf_unit_numel(ctypes.byref(cfg), unit))


class Model:
    """One sf_ctx: the layer-sliding training engine of one decoder."""

    def __init__(self, cfg: Config):
        self.cfg = cfg
        h = _VP()
        st = lib().sf_init_model(ctypes.byref(cfg), ctypes.byref(h))
        if st != SF_OK:
            raise SfError(st, "sf_init_model: " + lib().sf_last_error(None).decode(errors="replace"))
        self.h = h

    def close(self):
        if getattr(self, "h", None):
            lib().sf_free(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *a):
        self.close()

    def error(self) -> str:
        return lib().sf_last_error(self.h).decode(errors="replace")

    def numel(self, unit: int) -> int:
        return unit_numel(self.cfg, unit)

    def load(self, unit: int, master: np.ndarray):
        a = np.ascontiguousarray(master, dtype=np.float32).reshape(-1)
        _check(lib().sf_load_layer_weights(self.h, unit, a.ctypes.data, a.size), self.h,
               f"sf_load_layer_weights({unit})")

    def train_step(self, tokens: np.ndarray, labels: np.ndarray, adam: Adam | None = None) -> int:
        """Returns the status (raises on errors other than the ones asked about)."""
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        y = np.ascontiguousarray(labels, dtype=np.int32)
        assert t.shape == y.shape and t.ndim == 2
        st = lib().sf_train_step(self.h, t.ctypes.data, y.ctypes.data, t.shape[0], t.shape[1],
                                 ctypes.byref(adam) if adam is not None else None)
        return st

    def step(self, tokens, labels, adam: Adam | None = None) -> float:
        _check(self.train_step(tokens, labels, adam), self.h, "sf_train_step")
        return self.loss()

    def train_step_accum(self, tokens: np.ndarray, labels: np.ndarray,
                         adam: Adam | None = None) -> int:
        """One optimizer step over micro-batches: tokens, labels [n_micro, batch, seq].
        Returns the status."""
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        y = np.ascontiguousarray(labels, dtype=np.int32)
        assert t.shape == y.shape and t.ndim == 3
        return lib().sf_train_step_accum(self.h, t.ctypes.data, y.ctypes.data, t.shape[0],
                                         t.shape[1], t.shape[2],
                                         ctypes.byref(adam) if adam is not None else None)

    def step_accum(self, tokens, labels, adam: Adam | None = None) -> float:
        _check(self.train_step_accum(tokens, labels, adam), self.h, "sf_train_step_accum")
        return self.loss()

    def loss(self) -> float:
        out = _F32()
        _check(lib().sf_loss(self.h, ctypes.byref(out)), self.h, "sf_loss")
        return float(out.value)

    def adam_state(self, unit: int):
        """(m, v) of a unit as fp32 arrays in the caller's order."""
        m = np.empty(self.numel(unit), dtype=np.float32)
        v = np.empty_like(m)
        _check(lib().sf_get_adam_state(self.h, unit, m.ctypes.data, v.ctypes.data, m.size),
               self.h, "sf_get_adam_state")
        return m, v

    def set_adam_state(self, unit: int, m: np.ndarray, v: np.ndarray) -> None:
        m = np.ascontiguousarray(m, dtype=np.float32).reshape(-1)
        v = np.ascontiguousarray(v, dtype=np.float32).reshape(-1)
        _check(lib().sf_set_adam_state(self.h, unit, m.ctypes.data, v.ctypes.data, m.size),
               self.h, "sf_set_adam_state")

    @property
    def adam_step(self) -> int:
        t = _I64()
        _check(lib().sf_get_adam_step(self.h, ctypes.byref(t)), self.h, "sf_get_adam_step")
        return int(t.value)

    @adam_step.setter
    def adam_step(self, t: int) -> None:
        _check(lib().sf_set_adam_step(self.h, t), self.h, "sf_set_adam_step")

    def grads(self, unit: int) -> np.ndarray:
        out = np.empty(self.numel(unit), dtype=np.float32)
        _check(lib().sf_get_grads(self.h, unit, out.ctypes.data, out.size), self.h, "sf_get_grads")
        return out

    def weights(self, unit: int) -> np.ndarray:
        out = np.empty(self.numel(unit), dtype=np.float32)
        _check(lib().sf_get_weights(self.h, unit, out.ctypes.data, out.size), self.h, "sf_get_weights")
        return out

    def sync(self):
        """Wait for the host updates still running (async_update mode)."""
        _check(lib().sf_sync(self.h), self.h, "sf_sync")

    def set_timing(self, on: bool):
        _check(lib().sf_set_timing(self.h, 1 if on else 0), self.h, "sf_set_timing")

    def stats(self) -> dict:
        s = Stats()
        _check(lib().sf_get_stats(self.h, ctypes.byref(s)), self.h, "sf_get_stats")
        return s.as_dict()

    def trace(self, cap: int = 8192) -> list:
        """Host timeline records since the last call: (t_ms, kind name, unit)."""
        buf = (TraceEvent * cap)()
        n = _I32()
        _check(lib().sf_get_trace(self.h, buf, cap, ctypes.byref(n)), self.h, "sf_get_trace")
        return [(buf[i].t_ms, TRACE_KINDS.get(buf[i].kind, buf[i].kind), buf[i].unit) for i in range(n.value)]

    def inject(self, what: int, arg: int = 0):
        _check(lib().sf_debug_inject(self.h, what, arg), self.h, "sf_debug_inject")


# ------------------------------------------------------------------ kernel API
def _s(stream) -> int | None:
    return int(stream) if stream else None


def op_gemm(layout, epi, M, N, K, A, lda, B, ldb, C, ldc, R=0, ldr=0, alpha=1.0, stream=0) -> int:
    return lib().sf_op_gemm(layout, epi, M, N, K, A, lda, B, ldb, C, ldc, R or None, ldr, alpha, _s(stream))


def op_rmsnorm_fwd(x, g, y, rstd, rows, d, eps, stream=0) -> int:
    return lib().sf_op_rmsnorm_fwd(x, g, y, rstd, rows, d, eps, _s(stream))


def op_rmsnorm_bwd(x, g, rstd, dy, dres, dx, dxb, dg, scratch, rows, d, stream=0) -> int:
    return lib().sf_op_rmsnorm_bwd(x, g, rstd, dy, dres or None, dx, dxb, dg, scratch, rows, d, _s(stream))


def op_rmsnorm_bwd_noalloc(x, g, rstd, dy, dres, dx, dxb, dg, rows, d, stream=0) -> int:
    """sf_op_rmsnorm_bwd without a scratch argument (library-owned fixed array)."""
    return lib().sf_op_rmsnorm_bwd_noalloc(x, g, rstd, dy, dres or None, dx, dxb, dg, rows, d, _s(stream))


STATIC_SCRATCH_FLOATS = 4194304


def rmsnorm_bwd_scratch(rows, d) -> int:
    return int(lib().sf_op_rmsnorm_bwd_scratch(rows, d))


def rope_table(seq, head_dim, base) -> np.ndarray:
    out = np.empty((seq, head_dim // 2, 2), dtype=np.float32)
    _check(lib().sf_rope_table(seq, head_dim, base, out.ctypes.data), None, "sf_rope_table")
    return out


def op_rope(x, ld, tokens, seq, heads, head_dim, table, inverse=0, stream=0) -> int:
    return lib().sf_op_rope(x, ld, tokens, seq, heads, head_dim, table, inverse, _s(stream))


def op_attn_fwd(qkv, o, lse, B, S, Hq, Hkv, hd, stream=0) -> int:
    return lib().sf_op_attn_fwd(qkv, o, lse, B, S, Hq, Hkv, hd, _s(stream))


def lce_step(h_bf16: np.ndarray, w_bf16: np.ndarray, labels: np.ndarray,
             ignore_index: int = IGNORE_INDEX, model=None, dh_out=None, dw_out=None):
    """Fused LM head + cross-entropy on host arrays (uint16 bf16 bits):
    returns (loss, dh as uint16 bf16 bits [n, d], dw fp32 [v, d]).  dh_out
    and dw_out, if given, are contiguous arrays of those shapes and types
    that receive the gradients (page-locked ones let the copies run at the
    link's rate)."""
    h = np.ascontiguousarray(h_bf16, dtype=np.uint16)
    w = np.ascontiguousarray(w_bf16, dtype=np.uint16)
    y = np.ascontiguousarray(labels, dtype=np.int32).reshape(-1)
    n, d = h.shape
    v = w.shape[0]
    loss = _F32()
    dh = np.empty((n, d), dtype=np.uint16) if dh_out is None else dh_out
    dw = np.empty((v, d), dtype=np.float32) if dw_out is None else dw_out
    if dh.shape != (n, d) or dh.dtype != np.uint16 or not dh.flags.c_contiguous:
        raise ValueError("lce_step: dh_out must be a contiguous uint16 array of shape (n, d)")
    if dw.shape != (v, d) or dw.dtype != np.float32 or not dw.flags.c_contiguous:
        raise ValueError("lce_step: dw_out must be a contiguous float32 array of shape (v, d)")
    st = lib().sf_lce_step(model.h if model is not None else None, h.ctypes.data, w.ctypes.data,
                           y.ctypes.data, n, d, v, ignore_index, ctypes.byref(loss),
                           dh.ctypes.data, dw.ctypes.data)
    _check(st, model.h if model is not None else None, "sf_lce_step")
    return float(loss.value), dh, dw


def op_gemm_bias(M, N, K, A, lda, B, ldb, C, ldc, bias, alpha=1.0, stream=0) -> int:
    return lib().sf_op_gemm_bias(M, N, K, A, lda, B, ldb, C, ldc, bias, alpha, _s(stream))


def op_gemm_qkv(M, N, K, A, lda, B, ldb, C, ldc, bias, table, seq, rope_cols, head_dim,
                stream=0) -> int:
    """Q/K/V projection + optional bias + rotary embedding, one bf16 rounding."""
    return lib().sf_op_gemm_qkv(M, N, K, A, lda, B, ldb, C, ldc, bias or None, table, seq,
                                rope_cols, head_dim, _s(stream))


def op_gemm_swiglu(M, F, K, A, lda, B, ldb, m, ldm, ab=0, ldab=0, stream=0) -> int:
    """Gate/up projection with SwiGLU: m = silu(A Wg^T) * (A Wu^T), B = [Wg; Wu]."""
    return lib().sf_op_gemm_swiglu(M, F, K, A, lda, B, ldb, m, ldm, ab or None, ldab, _s(stream))


def op_gemm_swiglu_bwd(M, F, K, dy, lddy, wd, ldw, ab, ldab, dab, lddab, stream=0) -> int:
    """dm = dy wd through the SwiGLU backward into [da | db] (bf16)."""
    return lib().sf_op_gemm_swiglu_bwd(M, F, K, dy, lddy, wd, ldw, ab, ldab, dab, lddab, _s(stream))


def op_bias_grad(dy, ld, rows, cols, part, db, stream=0) -> int:
    return lib().sf_op_bias_grad(dy, ld, rows, cols, part, db, _s(stream))


def bias_grad_scratch_floats(rows, cols) -> int:
    return int(lib().sf_op_bias_grad_scratch(rows, cols))


def op_attn_bwd(qkv, o, dout, lse, delta, dq_acc, dqkv, B, S, Hq, Hkv, hd, table=0, stream=0,
                deterministic=0) -> int:
    return lib().sf_op_attn_bwd(qkv, o, dout, lse, delta, dq_acc, dqkv, B, S, Hq, Hkv, hd,
                                table or None, deterministic, _s(stream))


def attn_dq_scratch_floats(B, S, Hq, hd, deterministic=0) -> int:
    """Floats of the dq_acc scratch sf_op_attn_bwd needs."""
    return (((S + 127) // 128) if deterministic else 1) * B * S * Hq * hd


def op_swiglu_fwd(ab, m, rows, ffn, stream=0) -> int:
    return lib().sf_op_swiglu_fwd(ab, m, rows, ffn, _s(stream))


def op_swiglu_bwd(dm, ab, dab, rows, ffn, stream=0) -> int:
    return lib().sf_op_swiglu_bwd(dm, ab, dab, rows, ffn, _s(stream))


def lce_workspace_bytes(n, v, chunk_rows) -> int:
    return int(lib().sf_op_lce_workspace_bytes(n, v, chunk_rows))


def lce_launches() -> int:
    """Kernels launched by this thread's last successful op_lce call."""
    return int(lib().sf_op_lce_launches())


def op_lce(h, w, labels, n, d, v, n_valid, chunk_rows, workspace, loss, dh, dw, stream=0) -> int:
    return lib().sf_op_lce(h, w, labels, n, d, v, n_valid, chunk_rows, workspace, loss, dh, dw, _s(stream))


def probe_host_bandwidth(threads: int = 0, nbytes: int = 4 << 30) -> float:
    """GB/s of host memory traffic with the host Adam's access pattern."""
    out = ctypes.c_double()
    _check(lib().sf_probe_host_bandwidth(threads, nbytes, ctypes.byref(out)), None, "sf_probe_host_bandwidth")
    return out.value


def device_error() -> int:
    out = _I32()
    _check(lib().sf_op_device_error(ctypes.byref(out)), None, "sf_op_device_error")
    return int(out.value)
