"""Seeded synthetic inputs for the layer-sliding fine-tuning step.

Input generation only: nothing here computes any part of the training step.
Both sides of every parity check (the CPU oracle and the CUDA library) and the
benchmark draw weights, tokens and labels from this module, so the two sides
see bit-identical inputs.  The generator is defined in ``synth.c`` (a
counter-based SplitMix64 stream with a Box-Muller transform); ``*_np`` below
restate it in numpy so that the compiled copy can be checked against it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .configs import (ModelConfig, LceConfig, CONFIGS, LCE_STRESS, TEST_CONFIGS,
                      VARIANT_CONFIGS, IGNORE_INDEX, UNIT_EMBED, UNIT_FINAL_NORM, UNIT_LM_HEAD,
                      layer_tensor_shapes, unit_numel)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "_synth.so")
_lock = threading.Lock()
_lib = None

SEED_WEIGHTS = 1234
SEED_TOKENS = 42
SEED_IGNORE = 7


def build() -> str:
    """Compile synth.c into _synth.so (gcc, OpenMP).  Returns the path."""
    src = os.path.join(_HERE, "synth.c")
    tmp = _SO + ".tmp%d" % os.getpid()
    subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", src,
                           "-o", tmp, "-lm"])
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            src = os.path.join(_HERE, "synth.c")
            if (not os.path.exists(_SO)) or os.path.getmtime(_SO) < os.path.getmtime(src):
                build()
            lib = ctypes.CDLL(_SO)
            u64, i64, f64 = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double
            vp = ctypes.c_void_p
            lib.synth_normal_f32.argtypes = [u64, u64, u64, i64, f64, f64, vp]
            lib.synth_randint_i32.argtypes = [u64, u64, u64, i64, i64, vp]
            lib.synth_uniform_f64.argtypes = [u64, u64, u64, i64, vp]
            lib.synth_set_threads.argtypes = [ctypes.c_int]
            lib.synth_set_threads(int(os.environ.get("SYNTH_THREADS", "0")) or (os.cpu_count() or 1))
            _lib = lib
    return _lib


def normal(seed: int, stream: int, n: int, mean: float = 0.0, std: float = 1.0,
           offset: int = 0, out: np.ndarray | None = None) -> np.ndarray:
    """float32 draws mean + std * N(0,1), elements [offset, offset + n) of the stream."""
    if out is None:
        out = np.empty(n, dtype=np.float32)
    assert out.dtype == np.float32 and out.flags.c_contiguous and out.size == n
    _load().synth_normal_f32(seed, stream, offset, n, mean, std, out.ctypes.data)
    return out


def randint(seed: int, stream: int, n: int, hi: int, offset: int = 0) -> np.ndarray:
    """int32 draws uniform in [0, hi)."""
    out = np.empty(n, dtype=np.int32)
    _load().synth_randint_i32(seed, stream, offset, n, hi, out.ctypes.data)
    return out


def uniform(seed: int, stream: int, n: int, offset: int = 0) -> np.ndarray:
    """float64 draws uniform in [0, 1)."""
    out = np.empty(n, dtype=np.float64)
    _load().synth_uniform_f64(seed, stream, offset, n, out.ctypes.data)
    return out


# ---- numpy restatement of the generator (for cross-checking the C copy) ----
_M64 = np.uint64(0xFFFFFFFFFFFFFFFF)


def _sm64_np(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        z = z + np.uint64(0x9E3779B97F4A7C15)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        return z ^ (z >> np.uint64(31))


def _key_np(seed: int, stream: int) -> np.uint64:
    s = _sm64_np(np.array([stream + 1], dtype=np.uint64))[0]
    return _sm64_np(np.array([np.uint64(seed) ^ s], dtype=np.uint64))[0]


def _words_np(seed, stream, idx):
    with np.errstate(over="ignore"):
        return _sm64_np(_key_np(seed, stream) + idx.astype(np.uint64))


def uniform_np(seed, stream, n, offset=0):
    idx = np.arange(offset, offset + n, dtype=np.uint64)
    return (_words_np(seed, stream, idx) >> np.uint64(11)).astype(np.float64) * 2.0 ** -53


def normal_np(seed, stream, n, mean=0.0, std=1.0, offset=0):
    idx = np.arange(offset, offset + n, dtype=np.uint64)
    p = idx & ~np.uint64(1)
    u0 = (_words_np(seed, stream, p) >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
    u1 = (_words_np(seed, stream, p + np.uint64(1)) >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
    r = np.sqrt(-2.0 * np.log(1.0 - u0))
    phi = 2.0 * np.pi * u1
    z = np.where((idx & np.uint64(1)) == 1, r * np.sin(phi), r * np.cos(phi))
    return (mean + std * z).astype(np.float32)


def randint_np(seed, stream, n, hi, offset=0):
    v = np.floor(uniform_np(seed, stream, n, offset) * hi).astype(np.int64)
    return np.minimum(v, hi - 1).astype(np.int32)


# ---- workload inputs --------------------------------------------------------
def _stream(unit: int, tensor_idx: int) -> int:
    return (unit + 3) * 16 + tensor_idx


def layer_master(cfg: ModelConfig, layer: int, seed: int = SEED_WEIGHTS) -> np.ndarray:
    """fp32 master weights of decoder layer ``layer`` as one flat array, in the
    unit order g1, Wq, Wk, Wv, [bq, bk, bv,] Wo, g2, Wg, Wu, Wd (matrices and
    biases N(0, 0.02), gains 1)."""
    out = np.empty(unit_numel(cfg, layer), dtype=np.float32)
    off = 0
    for idx, (name, shape) in enumerate(layer_tensor_shapes(cfg)):
        n = int(np.prod(shape))
        if name in ("g1", "g2"):
            out[off:off + n] = 1.0
        else:
            normal(seed, _stream(layer, idx), n, 0.0, 0.02, out=out[off:off + n])
        off += n
    return out


def unit_master(cfg: ModelConfig, unit: int, seed: int = SEED_WEIGHTS) -> np.ndarray:
    """fp32 master weights for any unit: a layer index, UNIT_EMBED, UNIT_FINAL_NORM or UNIT_LM_HEAD."""
    if unit >= 0:
        return layer_master(cfg, unit, seed)
    n = unit_numel(cfg, unit)
    if n == 0:
        raise ValueError("unit %d has no tensor in this model" % unit)
    if unit == UNIT_FINAL_NORM:
        return np.ones(n, dtype=np.float32)
    return normal(seed, _stream(unit, 0), n, 0.0, 0.02)


def split_layer(cfg: ModelConfig, flat: np.ndarray) -> dict:
    """View a flat layer array as named tensors (no copy)."""
    out, off = {}, 0
    for name, shape in layer_tensor_shapes(cfg):
        n = int(np.prod(shape))
        out[name] = flat[off:off + n].reshape(shape)
        off += n
    assert off == flat.size
    return out


def tokens_and_labels(cfg: ModelConfig, seed: int = SEED_TOKENS):
    """Uniform token ids in [0, vocab); labels are the next token, the last
    position of each sequence is IGNORE_INDEX.  Shapes [batch, seq], int32."""
    tok = randint(seed, 0, cfg.batch * cfg.seq, cfg.vocab).reshape(cfg.batch, cfg.seq)
    lab = np.full_like(tok, IGNORE_INDEX)
    lab[:, :-1] = tok[:, 1:]
    return tok, lab


def lce_inputs(c: LceConfig, seed_w: int = SEED_WEIGHTS, seed_tok: int = SEED_TOKENS,
               seed_ign: int = SEED_IGNORE):
    """Final hidden states H ~ N(0,1) [n, d], LM-head weights N(0,0.02) [V, d]
    (both float32; round to bf16 on use), labels uniform in [0, V) with each
    position ignored with probability ``ignore_frac``."""
    n = c.batch * c.seq
    h = normal(seed_w, 900, n * c.hidden, 0.0, 1.0).reshape(n, c.hidden)
    w = normal(seed_w, 901, c.vocab * c.hidden, 0.0, 0.02).reshape(c.vocab, c.hidden)
    lab = randint(seed_tok, 1, n, c.vocab)
    ign = uniform(seed_ign, 2, n) < c.ignore_frac
    lab = np.where(ign, IGNORE_INDEX, lab).astype(np.int32)
    return h, w, lab
