"""Workload shapes for the layer-sliding fine-tuning step (shapes only)."""
from __future__ import annotations

from dataclasses import dataclass, replace

IGNORE_INDEX = -100
UNIT_EMBED = -1
UNIT_FINAL_NORM = -2
UNIT_LM_HEAD = -3


@dataclass(frozen=True)
class ModelConfig:
    name: str
    n_layers: int
    hidden: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    batch: int
    seq: int
    rms_eps: float = 1e-5
    rope_base: float = 10000.0
    ring_slots: int = 2
    qkv_bias: bool = False        # Qwen-style biases on the Q, K and V projections
    tie_embeddings: bool = False  # the LM head is the embedding matrix

    @property
    def tokens(self) -> int:
        return self.batch * self.seq

    def with_(self, **kw) -> "ModelConfig":
        return replace(self, **kw)


@dataclass(frozen=True)
class LceConfig:
    name: str
    hidden: int
    vocab: int
    batch: int
    seq: int
    ignore_frac: float = 0.1


def layer_tensor_shapes(c: ModelConfig):
    """(name, shape) of one decoder layer's tensors in unit order (the Q, K, V
    biases follow W_v when the model has them)."""
    q, kv = c.n_heads * c.head_dim, c.n_kv_heads * c.head_dim
    bias = [("bq", (q,)), ("bk", (kv,)), ("bv", (kv,))] if c.qkv_bias else []
    return [("g1", (c.hidden,)), ("wq", (q, c.hidden)), ("wk", (kv, c.hidden)),
            ("wv", (kv, c.hidden))] + bias + [
            ("wo", (c.hidden, q)), ("g2", (c.hidden,)),
            ("wg", (c.ffn, c.hidden)), ("wu", (c.ffn, c.hidden)), ("wd", (c.hidden, c.ffn))]


def unit_numel(c: ModelConfig, unit: int) -> int:
    if unit >= 0:
        n = 0
        for _, s in layer_tensor_shapes(c):
            k = 1
            for x in s:
                k *= x
            n += k
        return n
    if unit == UNIT_LM_HEAD and c.tie_embeddings:
        return 0  # no separate tensor
    if unit in (UNIT_EMBED, UNIT_LM_HEAD):
        return c.vocab * c.hidden
    if unit == UNIT_FINAL_NORM:
        return c.hidden
    raise ValueError(unit)


# The five workloads of the step (names follow their shapes).
CONFIGS = {
    "tiny": ModelConfig("tiny-2L-d256", 2, 256, 4, 4, 64, 688, 2048, 2, 128,
                        rope_base=10000.0, ring_slots=2),
    "1.3b": ModelConfig("1.3b-24L-d2048", 24, 2048, 16, 16, 64, 5504, 32000, 8, 1024,
                        rope_base=10000.0, ring_slots=2),
    "8b": ModelConfig("8b-32L-d4096-gqa", 32, 4096, 32, 8, 128, 14336, 128256, 8, 2048,
                      rope_base=500000.0, ring_slots=3),
    "123b-slice": ModelConfig("123b-slice-4L-d12288-gqa", 4, 12288, 96, 8, 128, 28672, 32768,
                              4, 1024, rope_base=10000.0, ring_slots=2),
}
LCE_STRESS = LceConfig("lce-d3584-v152064", 3584, 152064, 4, 4096, 0.1)

# Small shapes for element-by-element parity: several tiles plus ragged tails.
TEST_CONFIGS = {
    "small-gqa": ModelConfig("small-gqa-3L-d384", 3, 384, 6, 2, 64, 1000, 3000, 2, 200,
                             rope_base=10000.0, ring_slots=2),
    "small-hd128": ModelConfig("small-hd128-2L-d512", 2, 512, 4, 2, 128, 1368, 4000, 1, 300,
                               rope_base=500000.0, ring_slots=2),
    "micro": ModelConfig("micro-2L-d64", 2, 64, 2, 1, 32, 96, 50, 2, 8,
                         rope_base=10000.0, ring_slots=2),
    # Qwen-style: Q/K/V biases and an LM head tied to the embedding
    "small-qwen": ModelConfig("small-qwen-3L-d384", 3, 384, 6, 2, 64, 1000, 3000, 2, 200,
                              rope_base=1000000.0, ring_slots=2, qkv_bias=True,
                              tie_embeddings=True),
}

# A full-size model of that family: the Qwen2.5-3B shape (36 layers, hidden
# 2048, 16 query / 2 kv heads of 128, FFN 11008, vocab 151936, biases on
# Q/K/V, tied embeddings).
VARIANT_CONFIGS = {
    "qwen-3b": ModelConfig("qwen-3b-36L-d2048-gqa-tied", 36, 2048, 16, 2, 128, 11008, 151936,
                           8, 2048, rms_eps=1e-6, rope_base=1000000.0, ring_slots=3,
                           qkv_bias=True, tie_embeddings=True),
}
