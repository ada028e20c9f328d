"""CPU oracle for the layer-sliding fine-tuning step.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, links or runs
this package: only the tests, ``__graft_entry__.smoke()`` and the benchmark's
``cpu_baseline`` / ``--impl reference`` legs do.  It shares no code with the
CUDA library; the only thing both sides use is the seeded input generator in
``inputs/``.

The oracle is plain numpy: every step is written out from its textbook
definition, with numpy's matmul as the only library primitive, so that a
reader can check it against the definitions by eye.  It computes in float64
by default (``dtype=np.float32`` gives the fp32 variant that is timed as the
CPU baseline).

Parity status per function (all pinned; see tests/test_oracle_pins.py):
  rmsnorm_*        pinned: torch rms_norm + autograd, closed-form moment
  rope_*           pinned: complex-rotation form, relative-position property,
                   norm preservation, identity at position 0, worked values
  attention_*      pinned: torch scaled_dot_product_attention + autograd,
                   causal invariance, GQA == MHA with repeated K/V
  swiglu_*         pinned: torch silu + autograd, finite differences
  cross_entropy_*  pinned: torch cross_entropy, loss = ln V at zero logits,
                   gradient rows sum to zero, ignored rows zero
  step             pinned: torch autograd of an independently assembled model,
                   central finite differences in float64
  step_streamed    the same step with layer weights fetched one at a time
                   (step is built on it; pinned through step, and equal to
                   step bit for bit)
  adam_update      pinned: torch.optim.AdamW step, first-step closed form
  adam_update_bf16_states
                   pinned: unbiased stochastic rounding (mean over many
                   draws), exact on bf16 values, bits uniform; tracks
                   float32-state Adam over many steps where round-to-nearest
                   bf16 states stall
"""
from .llama_step import (  # noqa: F401
    IGNORE_INDEX, bf16_round, rmsnorm_fwd, rmsnorm_bwd, rope_tables, rope_fwd, rope_bwd,
    attention_fwd, attention_bwd, swiglu_fwd, swiglu_bwd, cross_entropy_fwd_bwd,
    layer_fwd, layer_bwd, step, step_streamed, adam_update, ModelWeights,
    lowbias32, sr_key, sr_bits, bf16_round_stochastic, adam_update_bf16_states)
